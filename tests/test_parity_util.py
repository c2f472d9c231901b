"""The parity harness itself, on the CPU: results made from the oracle's own
steps stand in for a device's, so that each acceptance rule of
``parity_util`` is seen to pass what it must pass and to fail what it must
fail -- a route flipped on an exact tie is checked against the oracle's
alternatives, a wrong output on a flipped query fails, a flip outside the
tie allowance fails, and a comparison with nothing compared fails."""
import numpy as np
import pytest
import torch

import oracle
import parity_util as pu
from mixture_top_attention_mita_b300 import synth


def _tied_case():
    # small-integer inputs: many queries have two landmarks with exactly the
    # same score, so a second route is as valid as the first
    w = synth.WORKLOADS["deit_t"].scaled(B=1, H=1)
    Q, K, V = synth.make_integer_inputs(w, seed=3)
    r = oracle.head(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io=w.dtype, debug=True)
    A = r["A"]
    tied = [q for q in range(w.N) if np.sum(A[q] == A[q].max()) > 1]
    assert tied, "the construction should give exact route ties"
    return w, Q, K, V, r, tied


def _gpu_like(w, r):
    out = torch.from_numpy(r["out"].copy()).to(synth.torch_dtype(w))
    return out, torch.from_numpy(r["idx"].copy()), torch.from_numpy(r["route"].copy())


def _flip(w, Q, K, V, r, out, route, q):
    """Route query q to its other tied landmark; its output is the oracle's
    output under that route."""
    A = r["A"][q]
    alt = [i for i in np.flatnonzero(A == A.max()) if i != r["route"][q]][0]
    route[q] = int(alt)
    o = oracle.attend_one(Q[0, 0][q], A, r["idx"][alt], K[0, 0], V[0, 0], r["Vl"], io=w.dtype)
    out[q] = torch.from_numpy(o).to(out.dtype)
    return alt


def test_identical_results_pass_directly():
    w, Q, K, V, r, _ = _tied_case()
    out, idx, route = _gpu_like(w, r)
    t = pu.Tally()
    pu.compare_head(w, Q[0, 0], K[0, 0], V[0, 0], out, idx, route, exact=True, tally=t)
    s = pu.check_tally(t, exact=True)
    assert s["direct_queries"] == w.N and s["unchecked_queries"] == 0 and s["max_abs"] < 1e-30


def test_tied_route_flip_is_checked_against_alternatives():
    w, Q, K, V, r, tied = _tied_case()
    out, idx, route = _gpu_like(w, r)
    for q in tied[:3]:
        _flip(w, Q, K, V, r, out, route, q)
    t = pu.Tally()
    pu.compare_head(w, Q[0, 0], K[0, 0], V[0, 0], out, idx, route, exact=False, tally=t)
    s = pu.check_tally(t, exact=False)
    assert s["alternative_checked"] == 3 and s["unchecked_queries"] == 0


def test_wrong_output_on_a_flipped_query_fails():
    w, Q, K, V, r, tied = _tied_case()
    out, idx, route = _gpu_like(w, r)
    q = tied[0]
    _flip(w, Q, K, V, r, out, route, q)
    out[q] += 0.5
    t = pu.Tally()
    pu.compare_head(w, Q[0, 0], K[0, 0], V[0, 0], out, idx, route, exact=False, tally=t)
    with pytest.raises(AssertionError):
        s = pu.check_tally(t, exact=False)
        assert s["max_abs"] <= pu.TOL[w.dtype][0]


def test_flip_on_exact_inputs_fails():
    w, Q, K, V, r, tied = _tied_case()
    out, idx, route = _gpu_like(w, r)
    _flip(w, Q, K, V, r, out, route, tied[0])
    with pytest.raises(AssertionError):
        pu.compare_head(w, Q[0, 0], K[0, 0], V[0, 0], out, idx, route, exact=True)


def test_route_outside_the_tie_allowance_fails():
    w = synth.WORKLOADS["deit_t"].scaled(B=1, H=1)
    Q, K, V = synth.make_inputs(w, seed=9)
    r = oracle.head(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io=w.dtype, debug=True)
    out, idx, route = _gpu_like(w, r)
    A = r["A"][0] / np.sqrt(w.d)
    worst = int(np.argmin(A))
    assert A.max() - A[worst] > pu.TIE_EPS
    route[0] = worst
    with pytest.raises(AssertionError):
        pu.compare_head(w, Q[0, 0], K[0, 0], V[0, 0], out, idx, route, exact=False)


def test_expert_outside_the_tie_allowance_fails():
    w = synth.WORKLOADS["deit_t"].scaled(B=1, H=1)
    Q, K, V = synth.make_inputs(w, seed=9)
    r = oracle.head(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io=w.dtype, debug=True)
    out, idx, route = _gpu_like(w, r)
    R = r["R"][0]
    outside = int(np.argmin(R))           # the worst key of landmark 0
    assert outside not in set(idx[0].tolist())
    row = sorted(set(idx[0].tolist()) - {int(idx[0][0])} | {outside})
    idx[0] = torch.tensor(row, dtype=idx.dtype)
    with pytest.raises(AssertionError):
        pu.compare_head(w, Q[0, 0], K[0, 0], V[0, 0], out, idx, route, exact=False)


def test_expert_alternatives_enumerate_the_tie_group():
    # keys 2, 3, 4 tie at the k-th score: every 2-of-3 choice beside key 0
    R = np.array([5.0, -1.0, 1.0, 1.0, 1.0, -2.0])
    alts = pu.expert_alternatives(R, np.array([0, 2, 3]), 3)
    assert sorted(tuple(a.tolist()) for a in alts) == [(0, 2, 3), (0, 2, 4), (0, 3, 4)]


def test_nothing_compared_fails():
    t = pu.Tally()
    with pytest.raises(AssertionError):
        pu.check_tally(t, exact=False)


def test_unchecked_share_is_bounded():
    t = pu.Tally()
    t.direct, t.unchecked = 90, 10
    t.add(np.zeros(4))
    with pytest.raises(AssertionError):
        pu.check_tally(t, exact=False)
