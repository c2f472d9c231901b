"""Comparison of the CUDA path's results with the CPU oracle.

Acceptance (per head):
  * expert indices and routes bit-exact on small-integer inputs;
  * on random inputs an expert may differ from the oracle's only by keys
    whose oracle score lies within 1e-4 (after the 1/sqrt(d) scale) of the
    oracle's k-th best score, and a route only to a landmark whose oracle
    score lies within 1e-4 of the best;
  * outputs: fp32 I/O max-abs <= 1e-5; bf16 I/O max-abs <= 2e-2 and
    mean-abs <= 1e-2.  A query whose route or routed expert agrees with the
    oracle's is compared with the oracle's output.  A query touched by an
    allowed near-tie flip is compared with the oracle's outputs for every
    choice the tie rule allows -- the routes within 1e-4 of the best, the
    experts that swap keys within 1e-4 of the k-th score -- all enumerated
    from the oracle's own scores, never from the GPU's choice; its output
    must match one of them.  Only a query with more allowed choices than
    ``MAX_ALTERNATIVES`` stays unchecked, and every call bounds how many do
    (none on integer inputs, where nothing may flip).
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch

import oracle

TIE_EPS = 1e-4
TOL = {"f32": (1e-5, 1e-5), "bf16": (2e-2, 1e-2)}
MAX_ALTERNATIVES = 64          # allowed (route, expert) choices enumerated per flipped query
MAX_UNCHECKED_SHARE = 0.01     # of the compared queries, on random inputs


def expert_alternatives(R_i, o_idx_i, k, cap=MAX_ALTERNATIVES):
    """Every expert the tie rule allows for one landmark: the oracle's set
    with any choice of the keys whose scaled score lies within TIE_EPS of the
    k-th best (``R_i`` scaled scores of the row).  None past ``cap``."""
    kth = np.sort(R_i)[::-1][k - 1]
    near = np.flatnonzero(np.abs(R_i - kth) < TIE_EPS)
    sure = sorted(set(int(j) for j in o_idx_i) - set(int(j) for j in near))
    need = k - len(sure)
    if math.comb(len(near), need) > cap:
        return None
    return [np.array(sorted(sure + list(c)), dtype=np.int32) for c in itertools.combinations(near, need)]


class Tally:
    """Counts over the heads of one comparison: queries compared directly,
    checked against enumerated alternatives, or left unchecked."""

    def __init__(self):
        self.direct = self.alternatives = self.unchecked = 0
        self.flipped_experts = 0
        self.diffs = []

    def add(self, d):
        self.diffs.append(d)

    def summary(self):
        d = np.concatenate(self.diffs) if self.diffs else np.zeros(0)
        return {"max_abs": float(d.max()) if d.size else 0.0, "mean_abs": float(d.mean()) if d.size else 0.0,
                "direct_queries": self.direct, "alternative_checked": self.alternatives,
                "unchecked_queries": self.unchecked, "flipped_experts": self.flipped_experts}


def _check_flipped(w, Qh, Kh, Vh, r, q_local, q_global, g_out_q, bad_alts, shared, scale):
    """Smallest max-abs distance between the GPU's output row and the
    oracle's output under every allowed (route, expert) choice of the query,
    or None when there are more than MAX_ALTERNATIVES choices."""
    A = r["A"][q_local]
    As = A * scale
    routes = np.flatnonzero(As >= As.max() - TIE_EPS)
    choices = []
    for rt in routes:
        alts = bad_alts.get(int(rt))
        experts = [r["idx"][rt]] if alts is None else alts
        if experts == "uncapped":
            return None
        choices += list(experts)
        if len(choices) > MAX_ALTERNATIVES:
            return None
    q = Qh[q_global]
    best = None
    for E in choices:
        o = oracle.attend_one(q, A, E, Kh, Vh, r["Vl"], io=w.dtype, shared=shared)
        dist = np.abs(g_out_q - o)
        if best is None or dist.max() < best.max():
            best = dist
    return best


def compare_head(w, Qh, Kh, Vh, out_h, idx_h, route_h, exact: bool, queries=None, tally=None, shared=True,
                 s=1, r=None):
    """Check one head.  Qh/Kh/Vh are the CPU input tensors [N, d]; out_h
    [nq, d], idx_h [m, k], route_h [nq] are the GPU results (CPU tensors)
    for the queries listed in ``queries`` (default all); ``shared=False``
    checks the routing-only variant, ``s > 1`` routing to s experts.
    ``r``: the oracle's result for this head, if already computed (with
    ``debug=True``)."""
    if r is None:
        r = oracle.head(Qh, Kh, Vh, w.grid, w.m, w.k, io=w.dtype, queries=queries, debug=True, shared=shared, s=s)
    tally = tally if tally is not None else Tally()
    scale = 1.0 / math.sqrt(w.d)
    g_idx = idx_h.numpy()
    g_route = route_h.numpy()
    o_idx, o_route = r["idx"], r["route"]
    assert g_idx.shape == o_idx.shape
    assert (np.diff(g_idx, axis=1) > 0).all(), "expert indices must be strictly ascending"
    assert ((g_idx >= 0) & (g_idx < w.N)).all()
    bad_alts = {}   # landmark -> allowed experts (or "uncapped")
    if exact:
        np.testing.assert_array_equal(g_idx, o_idx)
        np.testing.assert_array_equal(g_route, o_route)
    else:
        R = r["R"] * scale
        for i in np.flatnonzero((g_idx != o_idx).any(1)):
            kth = np.sort(R[i])[::-1][w.k - 1]
            diff = set(g_idx[i]) ^ set(o_idx[i])
            for j in diff:
                assert abs(R[i, j] - kth) < TIE_EPS, (i, j, R[i, j], kth)
            alts = expert_alternatives(R[i], o_idx[i], w.k)
            bad_alts[int(i)] = "uncapped" if alts is None else alts
        A = r["A"] * scale
        for q in np.flatnonzero(g_route != o_route):
            assert abs(A[q, g_route[q]] - A[q, o_route[q]]) < TIE_EPS, (q, g_route[q], o_route[q])
    tally.flipped_experts += len(bad_alts)
    ok = (g_route == o_route) & ~np.isin(o_route, list(bad_alts))
    if s > 1:
        # every one of the s experts must be the oracle's, and unflipped
        A = r["A"] * scale
        order = np.argsort(-A, axis=1, kind="stable")
        tops = order[:, :s]
        if s < w.m:
            gap = np.take_along_axis(A, order[:, s - 1:s], 1)[:, 0] - np.take_along_axis(A, order[:, s:s + 1], 1)[:, 0]
            ok &= exact | (gap >= TIE_EPS)
        ok &= ~np.isin(tops, list(bad_alts)).any(1)
    g_out = out_h.double().numpy()
    max_tol, mean_tol = TOL[w.dtype]
    assert np.isfinite(g_out).all()
    d = np.abs(g_out[ok] - r["out"][ok])
    tally.direct += int(ok.sum())
    if d.size:
        tally.add(d.ravel())
    qlist = np.arange(w.N) if queries is None else np.asarray(queries)
    for ql in np.flatnonzero(~ok):
        best = None
        if s == 1:
            best = _check_flipped(w, Qh, Kh, Vh, r, ql, int(qlist[ql]), g_out[ql], bad_alts, shared, scale)
        if best is None:
            tally.unchecked += 1
        else:
            tally.alternatives += 1
            tally.add(best)
    if exact:
        assert tally.unchecked == 0 and tally.alternatives == 0
    return r


def check_tally(tally, exact: bool, report=None):
    """Apply the output tolerances over everything compared, and bound the
    queries left unchecked."""
    summ = tally.summary()
    if report is not None:
        report.append(summ)
    compared = tally.direct + tally.alternatives
    total = compared + tally.unchecked
    assert compared > 0, "no output was compared"
    limit = 0 if exact else int(MAX_UNCHECKED_SHARE * total)
    assert tally.unchecked <= limit, f"{tally.unchecked} of {total} queries unchecked (limit {limit})"
    return summ


def compare_batch(w, Q, K, V, out, idx, route, exact: bool, heads=None, queries=None, report=None, shared=True,
                  s=1):
    """Check the listed (b, h) heads (default all) of a batch, then apply
    the tolerances and the unchecked-query bound over all of them."""
    out, idx, route = out.cpu(), idx.cpu(), route.cpu()
    if heads is None:
        heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    max_tol, mean_tol = TOL[w.dtype]
    tally = Tally()
    for b, h in heads:
        if queries is None:
            o, rt = out[b, h], route[b, h]
        else:
            qs = torch.as_tensor(queries, dtype=torch.long)
            o, rt = out[b, h][qs], route[b, h][qs]
        compare_head(w, Q[b, h], K[b, h], V[b, h], o, idx[b, h], rt, exact, queries=queries, tally=tally,
                     shared=shared, s=s)
    summ = check_tally(tally, exact, report)
    assert summ["max_abs"] <= max_tol, f"max-abs {summ['max_abs']:.3e} > {max_tol}"
    assert summ["mean_abs"] <= mean_tol, f"mean-abs {summ['mean_abs']:.3e} > {mean_tol}"
    return summ


def compare_long_head(w, Qh, Kh, Vh, out_q, idx_h, route_q, queries, exact=False, threads=None, report=None):
    """Check one long head on sampled queries with the threaded oracle
    driver (every landmark row, the listed queries): experts of every
    landmark under the tie rule, routes and outputs of the sampled queries
    (flipped ones against the oracle's enumerated alternatives)."""
    r = oracle.head_threaded(Qh, Kh, Vh, w.grid, w.m, w.k, io=w.dtype, queries=queries, threads=threads)
    scale = 1.0 / math.sqrt(w.d)
    g_idx, g_route, g_out = idx_h.numpy(), route_q.numpy(), out_q.double().numpy()
    assert (np.diff(g_idx, axis=1) > 0).all() and ((g_idx >= 0) & (g_idx < w.N)).all()
    assert np.isfinite(g_out).all()
    bad_alts = {}
    for i in np.flatnonzero((g_idx != r["idx"]).any(1)):
        assert not exact, f"expert {i} differs on exact inputs"
        Ri = oracle.scores_row(r["Ql"][i], Kh) * scale
        kth = r["kth"][i] * scale
        for j in set(g_idx[i]) ^ set(r["idx"][i]):
            assert abs(Ri[j] - kth) < TIE_EPS, (i, j, Ri[j], kth)
        alts = expert_alternatives(Ri, r["idx"][i], w.k)
        bad_alts[int(i)] = "uncapped" if alts is None else alts
    As = r["A"] * scale
    for q in np.flatnonzero(g_route != r["route"]):
        assert not exact, f"route of query {queries[q]} differs on exact inputs"
        assert abs(As[q, g_route[q]] - As[q, r["route"][q]]) < TIE_EPS
    ok = (g_route == r["route"]) & ~np.isin(r["route"], list(bad_alts))
    tally = Tally()
    tally.flipped_experts = len(bad_alts)
    tally.direct = int(ok.sum())
    tally.add(np.abs(g_out[ok] - r["out"][ok]).ravel())
    for ql in np.flatnonzero(~ok):
        best = _check_flipped(w, Qh, Kh, Vh, r, ql, int(queries[ql]), g_out[ql], bad_alts, True, scale)
        if best is None:
            tally.unchecked += 1
        else:
            tally.alternatives += 1
            tally.add(best)
    summ = check_tally(tally, exact, report)
    max_tol, mean_tol = TOL[w.dtype]
    assert summ["max_abs"] <= max_tol, f"max-abs {summ['max_abs']:.3e} > {max_tol}"
    assert summ["mean_abs"] <= mean_tol, f"mean-abs {summ['mean_abs']:.3e} > {mean_tol}"
    return summ
