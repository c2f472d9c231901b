"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a library routine, brute force,
a closed form, an invariant or a value printed in the method description
(36Kr / 新智元 "注意力也是FFN？" and its English version).  Planted-mistake
tests at the end show that a plausible slip in the oracle fails a pin.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from mixture_top_attention_mita_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (scale * torch.randn(*shape, generator=g, dtype=torch.float64)).numpy()


# ---------------------------------------------------------------- rounding
def test_round_bf16_matches_torch_on_fp32_values():
    # torch rounds fp32 -> bf16 to nearest, ties to even; on fp32-representable
    # inputs (single rounding) the oracle must agree bit for bit.
    g = torch.Generator("cpu").manual_seed(3)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-20, 20, (20000,), generator=g).float())
    # include exact midpoints between bf16 neighbours
    mids = (torch.randn(2000, generator=g).to(torch.bfloat16).float().view(torch.int32) + (1 << 15)).view(torch.float32)
    x = torch.cat([x, mids])
    ref = x.to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in x.double().numpy()])
    assert np.array_equal(ref, got)


def test_round_bf16_hand_cases():
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0                 # tie -> even (down)
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6     # tie -> even (up)
    assert oracle.round_bf16(-(1 + 2 ** -8)) == -1.0
    assert oracle.round_bf16(1 + 2 ** -8 + 2 ** -30) == 1 + 2 ** -7  # above the midpoint
    assert oracle.round_bf16(0.0) == 0.0


# ---------------------------------------------------------------- pooling
@pytest.mark.parametrize("gh,gw,ph,pw", [(14, 14, 5, 5), (56, 56, 7, 7), (1, 512, 1, 8),
                                         (7, 9, 3, 4), (5, 5, 5, 5), (6, 6, 1, 1)])
def test_pool_matches_adaptive_avg_pool2d(gh, gw, ph, pw):
    N, d, m = gh * gw, 8, ph * pw
    Q = _rand((N, d), 11)
    r = oracle.head(Q, Q, Q, (gh, gw, ph, pw), m, 1, io="f64", debug=True)
    ref = F.adaptive_avg_pool2d(torch.from_numpy(Q).T.reshape(1, d, gh, gw), (ph, pw))
    ref = ref.reshape(d, m).T.numpy()
    np.testing.assert_allclose(r["Ql"], ref, rtol=0, atol=1e-13)


def test_pool_bins_14_to_5_overlap():
    # The 14 -> 5 adaptive bins overlap; their union covers every row once or twice.
    bins = [oracle.pool_bin(i, 14, 5) for i in range(5)]
    cover = np.zeros(14, int)
    for lo, hi in bins:
        cover[lo:hi] += 1
    assert cover.min() == 1 and cover.max() == 2
    assert bins[0][0] == 0 and bins[-1][1] == 14


def test_pool_bf16_rounds_the_exact_mean():
    # Q_l in the bf16 pipeline is the bf16 rounding of the exact fp64 mean.
    Q = torch.randn(196, 16, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    f = oracle.head(Q, Q, Q, (14, 14, 5, 5), 25, 3, io="f64", debug=True)["Ql"]
    b = oracle.head(Q, Q, Q, (14, 14, 5, 5), 25, 3, io="bf16", debug=True)["Ql"]
    np.testing.assert_array_equal(b, np.vectorize(oracle.round_bf16)(f))


def _bf16_nearest(x):
    """Nearest bf16 value to the rational x, ties to the even significand:
    written here from the format's definition (8 significant bits), with
    exact fractions, independently of the oracle's rounding routine."""
    from fractions import Fraction
    if x == 0:
        return Fraction(0)
    sign, a = (-1, -x) if x < 0 else (1, x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 7)               # spacing of bf16 values in [2^e, 2^(e+1))
    lo = (a // ulp) * ulp
    rem = a - lo
    if rem * 2 > ulp or (rem * 2 == ulp and (lo / ulp) % 2 == 1):
        lo += ulp
    return sign * lo


@pytest.mark.parametrize("count_grid", [(3, 4), (4, 4)])
def test_pool_bf16_rounds_exact_rational_means_at_midpoints(count_grid):
    # One bin of 12 or 16 tokens.  Each feature's values are integers below
    # 256 (exact in bf16) whose sum puts the exact mean on a bf16 rounding
    # midpoint (k + 1/2 for a mean in [128, 256)), or a 2^-20 value shifts
    # the sum just above or just below that midpoint.  The landmark must be
    # the bf16 value nearest to the exact rational mean: ties to even on the
    # midpoint, away from it otherwise.
    from fractions import Fraction
    gh, gw = count_grid
    n = gh * gw
    rng = np.random.default_rng(n)
    d = 48
    Q = np.zeros((n, d))
    for f in range(d):
        kind = f % 3
        k = int(rng.integers(128, 220))          # keeps every value below 256
        target = n * k + n // 2                      # n * (k + 1/2)
        free = n - 1 if kind else n                  # one token carries the 2^-20 shift
        vals = np.full(free, target // free)
        vals[: target - vals.sum()] += 1
        rng.shuffle(vals)
        Q[:free, f] = vals
        if kind:
            Q[n - 1, f] = 2.0 ** -20 if kind == 1 else -(2.0 ** -20)
    assert (np.abs(Q) < 256).all()
    Qb = torch.from_numpy(Q).to(torch.bfloat16)
    assert np.array_equal(Qb.double().numpy(), Q)    # every value exact in bf16
    r = oracle.head(Qb, Qb, Qb, (gh, gw, 1, 1), 1, 1, io="bf16", debug=True)
    want = [float(_bf16_nearest(sum(Fraction(float(v)) for v in Q[:, f]) / n)) for f in range(d)]
    np.testing.assert_array_equal(r["Ql"][0], want)
    means = Q.sum(0) / n
    assert (np.round(means[0::3] * 2) % 2 == 1).all()   # the tie features sit on midpoints


# ---------------------------------------------------------------- top-k
def _brute_topk(R, k):
    # j is selected iff fewer than k keys beat it, where l beats j when
    # R[l] > R[j], or R[l] == R[j] and l < j.
    m, N = R.shape
    out = []
    for i in range(m):
        sel = []
        for j in range(N):
            beat = sum(1 for l in range(N) if R[i, l] > R[i, j] or (R[i, l] == R[i, j] and l < j))
            if beat < k:
                sel.append(j)
        out.append(sel)
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("k", [1, 5, 17, 36])
def test_topk_brute_force_with_ties(k):
    g = torch.Generator().manual_seed(k)
    Q = torch.randint(-2, 3, (36, 4), generator=g).double().numpy()
    K = torch.randint(-1, 2, (36, 4), generator=g).double().numpy()   # many exact ties
    r = oracle.head(Q, K, K, (6, 6, 2, 3), 6, k, io="f64", debug=True)
    np.testing.assert_array_equal(r["idx"], _brute_topk(r["R"], k))


def test_scores_match_matmul():
    Q, K = _rand((49, 8), 1), _rand((49, 8), 2)
    r = oracle.head(Q, K, K, (7, 7, 2, 2), 4, 5, io="f64", debug=True)
    np.testing.assert_allclose(r["R"], r["Ql"] @ K.T, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["A"], Q @ r["Ql"].T, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- route
def test_route_is_first_argmax():
    g = torch.Generator().manual_seed(9)
    Q = torch.randint(-1, 2, (64, 4), generator=g).double().numpy()
    r = oracle.head(Q, Q, Q, (8, 8, 4, 4), 16, 3, io="f64", debug=True)
    A = Q @ r["Ql"].T
    for q in range(64):
        best = np.flatnonzero(A[q] == A[q].max())
        assert r["route"][q] == best[0]
    assert (np.sum(A == A.max(1, keepdims=True), 1) > 1).any()  # ties were exercised


# ---------------------------------------------------------------- values and output
def test_landmark_values_match_sdpa():
    Q, K, V = _rand((196, 16), 1), _rand((196, 16), 2), _rand((196, 16), 3)
    r = oracle.head(Q, K, V, (14, 14, 5, 5), 25, 25, io="f64", debug=True)
    t = torch.from_numpy
    ref = F.scaled_dot_product_attention(t(r["Ql"])[None], t(K)[None], t(V)[None])[0].numpy()
    np.testing.assert_allclose(r["Vl"], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("grid,m,k,d", [((14, 14, 5, 5), 25, 25, 16), ((8, 8, 2, 4), 8, 9, 8),
                                        ((1, 96, 1, 6), 6, 40, 12)])
def test_output_matches_masked_sdpa(grid, m, k, d):
    N = grid[0] * grid[1]
    Q, K, V = _rand((N, d), 4), _rand((N, d), 5), _rand((N, d), 6)
    r = oracle.head(Q, K, V, grid, m, k, io="f64", debug=True)
    keys = np.concatenate([r["Ql"], K])
    vals = np.concatenate([r["Vl"], V])
    mask = np.zeros((N, m + N), bool)
    mask[:, :m] = True
    for q in range(N):
        mask[q, m + r["idx"][r["route"][q]]] = True
    t = torch.from_numpy
    ref = F.scaled_dot_product_attention(t(Q)[None], t(keys)[None], t(vals)[None],
                                         attn_mask=t(mask)[None])[0].numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-12)


def test_full_attention_special_case():
    # k = N and m = 1: one landmark (the mean query) and every key routed, so
    # the operator is textbook attention over N + 1 keys [Q_l ; K].
    N, d = 48, 8
    Q, K, V = _rand((N, d), 7), _rand((N, d), 8), _rand((N, d), 9)
    r = oracle.head(Q, K, V, (6, 8, 1, 1), 1, N, io="f64", debug=True)
    np.testing.assert_allclose(r["Ql"][0], Q.mean(0), rtol=0, atol=1e-14)
    assert (r["route"] == 0).all() and (r["idx"][0] == np.arange(N)).all()
    t = torch.from_numpy
    vl = F.scaled_dot_product_attention(t(Q.mean(0, keepdims=True))[None], t(K)[None], t(V)[None])[0]
    ref = F.scaled_dot_product_attention(t(Q)[None], torch.cat([t(Q.mean(0, keepdims=True)), t(K)])[None],
                                         torch.cat([vl, t(V)])[None])[0].numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("grid,m,k,d", [((14, 14, 5, 5), 25, 25, 16), ((1, 96, 1, 6), 6, 40, 12)])
def test_routing_only_matches_masked_sdpa(grid, m, k, d):
    # Routing-only variant (the article's ablation without the shared expert):
    # each query attends to its expert's k keys alone.
    N = grid[0] * grid[1]
    Q, K, V = _rand((N, d), 14), _rand((N, d), 15), _rand((N, d), 16)
    r = oracle.head(Q, K, V, grid, m, k, io="f64", debug=True, shared=False)
    mask = np.zeros((N, N), bool)
    for q in range(N):
        mask[q, r["idx"][r["route"][q]]] = True
    t = torch.from_numpy
    ref = F.scaled_dot_product_attention(t(Q)[None], t(K)[None], t(V)[None], attn_mask=t(mask)[None])[0].numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-12)
    W = r["W"]
    assert (W[:, :m] == 0).all() and (W[:, m:] > 0).all()
    np.testing.assert_allclose(W.sum(1), 1.0, rtol=0, atol=1e-12)


def test_routing_only_full_attention_special_case():
    # k = N, m = 1, routing only: every key is routed and nothing else takes
    # part, so the operator is textbook attention over the N keys.
    N, d = 48, 8
    Q, K, V = _rand((N, d), 17), _rand((N, d), 18), _rand((N, d), 19)
    r = oracle.head(Q, K, V, (6, 8, 1, 1), 1, N, io="f64", shared=False)
    t = torch.from_numpy
    ref = F.scaled_dot_product_attention(t(Q)[None], t(K)[None], t(V)[None])[0].numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-12)


def _top_s_reference(Q, K, V, r, m, s):
    """Masked SDPA over [Q_l ; K]: every shared pair, and the keys of the s best
    experts of each query (stable order on -A: ties to the lower landmark)."""
    N = Q.shape[0]
    top = np.argsort(-r["A"], axis=1, kind="stable")[:, :s]
    mask = np.zeros((N, m + N), bool)
    mask[:, :m] = True
    for q in range(N):
        for e in top[q]:
            mask[q, m + r["idx"][e]] = True
    t = torch.from_numpy
    keys, vals = np.concatenate([r["Ql"], K]), np.concatenate([r["Vl"], V])
    return F.scaled_dot_product_attention(t(Q)[None], t(keys)[None], t(vals)[None], attn_mask=t(mask)[None])[0].numpy()


@pytest.mark.parametrize("s", [2, 3, 25])
def test_top_s_routing_matches_masked_sdpa(s):
    # s > 1: the union of the s best experts' keys, each key once, next to the
    # m shared pairs in one softmax.
    Q, K, V = _rand((196, 16), 21), _rand((196, 16), 22), _rand((196, 16), 23)
    r = oracle.head(Q, K, V, (14, 14, 5, 5), 25, 25, io="f64", debug=True, s=s)
    np.testing.assert_allclose(r["out"], _top_s_reference(Q, K, V, r, 25, s), rtol=0, atol=1e-12)


def test_top_s_routing_ties_on_integer_inputs():
    # small-integer inputs: many exactly tied query-landmark scores, so the
    # tie rule (lower landmark first) decides which experts join
    g = torch.Generator("cpu").manual_seed(24)
    Q = torch.randint(-1, 2, (64, 8), generator=g).double().numpy()
    K = torch.randint(-2, 3, (64, 8), generator=g).double().numpy()
    V = torch.randint(-3, 4, (64, 8), generator=g).double().numpy()
    r = oracle.head(Q, K, V, (8, 8, 2, 4), 8, 6, io="f64", debug=True, s=3)
    A = r["A"]
    assert any(len(np.unique(row)) < len(row) for row in A)   # ties present
    np.testing.assert_allclose(r["out"], _top_s_reference(Q, K, V, r, 8, 3), rtol=0, atol=1e-12)


def _fd_check(grid, m, k, d, shared, seed):
    """Central finite differences of L = sum(out * G) against the oracle's
    backward (fp64, no rounding), with the experts and routes checked to be
    the same at every perturbed point."""
    N = grid[0] * grid[1]
    Q, K, V = _rand((N, d), seed), _rand((N, d), seed + 1), _rand((N, d), seed + 2)
    G = _rand((N, d), seed + 3)
    base = oracle.head(Q, K, V, grid, m, k, io="f64", shared=shared)
    dQ, dK, dV = oracle.backward(Q, K, V, G, grid, m, k, io="f64", shared=shared)
    eps = 1e-6
    for X, dX in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        for a in range(N):
            for b in range(d):
                old = X[a, b]
                X[a, b] = old + eps
                rp = oracle.head(Q, K, V, grid, m, k, io="f64", shared=shared)
                X[a, b] = old - eps
                rm = oracle.head(Q, K, V, grid, m, k, io="f64", shared=shared)
                X[a, b] = old
                for rr in (rp, rm):
                    assert (rr["idx"] == base["idx"]).all() and (rr["route"] == base["route"]).all()
                num[a, b] = ((rp["out"] * G).sum() - (rm["out"] * G).sum()) / (2 * eps)
        np.testing.assert_allclose(dX, num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("grid,m,k,d,shared", [((6, 6, 2, 3), 6, 5, 4, True), ((1, 20, 1, 4), 4, 7, 3, True),
                                               ((6, 6, 2, 3), 6, 5, 4, False), ((5, 5, 2, 3), 6, 5, 3, True)])
def test_backward_matches_finite_differences(grid, m, k, d, shared):
    # The backward pass: the experts and routes are constants; gradients flow
    # through both softmaxes, the landmark values and the pooling (the 5 x 5
    # grid into 2 x 3 bins has overlapping bins, so some tokens feed two or
    # four landmarks).
    _fd_check(grid, m, k, d, shared, seed=31)


def _golden_keys_per_query():
    rows = []
    with open(os.path.join(GOLDEN, "keys_per_query.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                m, k, total, _ = line.split()
                rows.append((int(m), int(k), int(total)))
    return rows


@pytest.mark.parametrize("m,k,total", _golden_keys_per_query())
def test_keys_per_query_printed_value(m, k, total):
    # m shared + k routed entries per query (25+25=50, 49+49=98 as printed).
    side = int(math.isqrt(m))
    grid = (side * 4, side * 4, side, side)
    N = grid[0] * grid[1]
    Q, K, V = _rand((N, 8), 1), _rand((N, 8), 2), _rand((N, 8), 3)
    r = oracle.head(Q, K, V, grid, m, k, io="f64", debug=True)
    W = r["W"]
    assert W.shape[1] == total
    assert (W > 0).sum(1).min() == total        # every entry takes part
    np.testing.assert_allclose(W.sum(1), 1.0, rtol=0, atol=1e-12)


def test_weights_sum_to_one_and_shift_invariance():
    Q, K, V = _rand((196, 8), 1), _rand((196, 8), 2), _rand((196, 8), 3)
    g = (14, 14, 5, 5)
    r0 = oracle.head(Q, K, V, g, 25, 25, io="f64", debug=True)
    np.testing.assert_allclose(r0["W"].sum(1), 1.0, rtol=0, atol=1e-12)
    c = np.linspace(-3, 3, 8)
    r1 = oracle.head(Q, K, V + c, g, 25, 25, io="f64")
    np.testing.assert_allclose(r1["out"], r0["out"] + c, rtol=0, atol=1e-12)


def test_feature_permutation_equivariance():
    Q, K, V = _rand((196, 8), 1), _rand((196, 8), 2), _rand((196, 8), 3)
    p = np.random.default_rng(0).permutation(8)
    g = (14, 14, 5, 5)
    r0 = oracle.head(Q, K, V, g, 25, 25, io="f64")
    r1 = oracle.head(Q[:, p], K[:, p], V[:, p], g, 25, 25, io="f64")
    np.testing.assert_array_equal(r0["idx"], r1["idx"])
    np.testing.assert_array_equal(r0["route"], r1["route"])
    np.testing.assert_allclose(r1["out"], r0["out"][:, p], rtol=0, atol=1e-12)


def test_experts_distinct_sorted_and_overlapping():
    w = synth.WORKLOADS["deit_s"].scaled(B=1, H=1)
    Q, K, V = synth.make_inputs(w)
    r = oracle.head(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io="bf16")
    idx = r["idx"]
    assert (np.diff(idx, axis=1) > 0).all()
    assert len(np.unique(idx)) < idx.size      # experts overlap on clustered tokens


def test_query_subset_matches_full():
    Q, K, V = _rand((196, 8), 1), _rand((196, 8), 2), _rand((196, 8), 3)
    g = (14, 14, 5, 5)
    full = oracle.head(Q, K, V, g, 25, 25, io="bf16")
    qs = [195, 0, 77]
    sub = oracle.head(Q, K, V, g, 25, 25, io="bf16", queries=qs)
    np.testing.assert_array_equal(sub["out"], full["out"][qs])
    np.testing.assert_array_equal(sub["route"], full["route"][qs])


def test_batch_forward_matches_heads():
    w = synth.WORKLOADS["deit_t"].scaled(B=2, H=2)
    Q, K, V = synth.make_inputs(w)
    r = oracle.forward(Q, K, V, w.grid, w.m, w.k, io="bf16")
    h = oracle.head(Q[1, 0], K[1, 0], V[1, 0], w.grid, w.m, w.k, io="bf16")
    np.testing.assert_array_equal(r["out"][1, 0], h["out"])
    np.testing.assert_array_equal(r["idx"][1, 0], h["idx"])


def test_integer_inputs_have_exact_bf16_means():
    for name in ("deit_s", "hires56", "long1d"):
        w = synth.WORKLOADS[name]
        w = w.scaled(B=1, H=1, N=w.gh * w.gw if w.gh > 1 else 2048,
                     gw=w.gw if w.gh > 1 else 2048, pw=w.pw if w.gh > 1 else 8, m=w.m if w.gh > 1 else 8)
        Q, K, V = synth.make_integer_inputs(w)
        f = oracle.head(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, 3, io="f64", debug=True)["Ql"]
        np.testing.assert_array_equal(f, np.vectorize(oracle.round_bf16)(f))


# ---------------------------------------------------------------- planted mistakes
_MUTANTS = {
    "drop_shared_values": ("for (int i = 0; i < m; ++i) s += logit[i] * Vl[(size_t)i * d + f];", ""),
    "unscaled_routed_logit": ("logit[m + t] = s * scale;", "logit[m + t] = s;"),
    "ties_to_higher_index": ("return (ia > ib) - (ia < ib);", "return (ia < ib) - (ia > ib);"),
    # bf16 rounding with ties away from zero instead of to even
    "bf16_ties_away": ("double r = nearbyint(y);", "double r = round(y);"),
    "pool_bins_floor_end": ("*hi = ((i + 1) * G + P - 1) / P;", "*hi = ((i + 1) * G) / P;"),
    "route_last_argmax": ("if (s > A[best]) best = i;", "if (s >= A[best]) best = i;"),
    "values_wrong_row": ("acc[f] += w * V[(size_t)j * d + f];", "acc[f] += w * V[(size_t)(N - 1 - j) * d + f];"),
    "routing_only_keeps_shared": ("logit[i] = shared ? A[i] * scale : -INFINITY;", "logit[i] = A[i] * scale;"),
    "top_s_first_expert_only": ("for (int r = 0; r < s; ++r)\n        for (int t = 0; t < k; ++t) in_union",
                                "for (int r = 0; r < 1; ++r)\n        for (int t = 0; t < k; ++t) in_union"),
    "top_s_ties_to_higher": ("if (!taken && (best < 0 || A[i] > A[best])) best = i;",
                             "if (!taken && (best < 0 || A[i] >= A[best])) best = i;"),
    "backward_softmax_sign": ("for (int l = 0; l < m + k; ++l) dl[l] = w[l] * (dl[l] - wdw);",
                              "for (int l = 0; l < m + k; ++l) dl[l] = w[l] * (dl[l] + wdw);"),
    "backward_pool_count": ("dQ[(size_t)(y * gw + x) * d + f] += src[f] / count;",
                            "dQ[(size_t)(y * gw + x) * d + f] += src[f];"),
    "backward_values_transpose": ("dV[(size_t)j * d + f] += pij * dVl[(size_t)i * d + f];",
                                  "dV[(size_t)j * d + f] += pij * dVl[(size_t)((i + 1) % m) * d + f];"),
    # the bins taken as a partition (floor bounds) in the pool backward: the
    # same as the adaptive bins unless bins overlap
    "backward_pool_partition": ("            for (int y = r0; y < r1; ++y)\n"
                                "                for (int x = c0; x < c1; ++x)\n"
                                "                    for (int f = 0; f < d; ++f) dQ[",
                                "            for (int y = r * gh / ph; y < (r + 1) * gh / ph; ++y)\n"
                                "                for (int x = c * gw / pw; x < (c + 1) * gw / pw; ++x)\n"
                                "                    for (int f = 0; f < d; ++f) dQ["),
}


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    """A copy of the oracle source with one plausible slip planted in it must
    fail at least one of the pins above."""
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mita_oracle.c")).read()
    a, b = _MUTANTS[name]
    assert a in src
    c = tmp_path / "mutant.c"
    c.write_text(src.replace(a, b))
    so = tmp_path / "mutant.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", str(so), str(c), "-lm"])
    pins = [lambda: test_output_matches_masked_sdpa((8, 8, 2, 4), 8, 9, 8),
            lambda: test_landmark_values_match_sdpa(),
            lambda: test_topk_brute_force_with_ties(17),
            lambda: test_route_is_first_argmax(),
            lambda: test_pool_matches_adaptive_avg_pool2d(14, 14, 5, 5),
            lambda: test_pool_bf16_rounds_exact_rational_means_at_midpoints((3, 4)),
            lambda: test_routing_only_full_attention_special_case(),
            lambda: test_top_s_routing_matches_masked_sdpa(3),
            lambda: test_top_s_routing_ties_on_integer_inputs(),
            lambda: _fd_check((6, 6, 2, 3), 6, 5, 4, True, seed=31),
            lambda: _fd_check((5, 5, 2, 3), 6, 5, 3, True, seed=31)]
    failures = 0
    with oracle.swapped_library(str(so)):
        for pin in pins:
            try:
                pin()
            except AssertionError:
                failures += 1
    assert failures >= 1, name


def test_threaded_driver_matches_head():
    # The long-sequence parity tests run the same oracle steps landmark row
    # by landmark row over host threads; the results must be head()'s, bit
    # for bit, and scores_row / attend_one must restate head()'s rows.
    w = synth.WORKLOADS["long1d"].scaled(B=1, H=1, N=4096, gw=4096, pw=16, m=16, k=100)
    Q, K, V = synth.make_inputs(w)
    a = oracle.head(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io="bf16", debug=True)
    qs = [0, 5, 2047, 4095]
    b = oracle.head_threaded(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io="bf16", queries=qs, threads=4)
    for key in ("idx", "Ql", "Vl"):
        np.testing.assert_array_equal(a[key], b[key])
    np.testing.assert_array_equal(a["out"][qs], b["out"])
    np.testing.assert_array_equal(a["route"][qs], b["route"])
    np.testing.assert_array_equal(a["A"][qs], b["A"])
    np.testing.assert_array_equal(np.sort(a["R"], 1)[:, ::-1][:, w.k - 1], b["kth"])
    np.testing.assert_array_equal(oracle.scores_row(a["Ql"][3], K[0, 0]), a["R"][3])
    q = 5
    o = oracle.attend_one(Q[0, 0][q], a["A"][q], a["idx"][a["route"][q]], K[0, 0], V[0, 0], a["Vl"], io="bf16")
    np.testing.assert_array_equal(o, a["out"][q])
