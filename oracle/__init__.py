"""MiTA forward oracle -- test infrastructure only.

A slow, single-threaded fp64 CPU restatement of the Mixture-of-Top-k
Attention forward operator (36Kr / 新智元 "注意力也是FFN？", section
"用少量地标查询，同时构造全局概括与细节专家"; English version "Is Attention Also
FFN?", section "Construct global generalization and detail experts ...").
The arithmetic lives in ``mita_oracle.c``; this module compiles it with gcc
and marshals numpy arrays to it.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library neither imports nor
links it, and it shares no code with the CUDA library.

Parity status per function: every function is pinned by a ``-m "not gpu"``
test in ``tests/test_oracle_pins.py`` against something other than itself
(library routines, brute force, closed forms, invariants).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mita_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

IO_F64, IO_F32, IO_BF16 = 0, 1, 2
_IO_NAMES = {"f64": IO_F64, "f32": IO_F32, "bf16": IO_BF16}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``mita_oracle.c`` into ``liboracle.so`` next to it (IEEE fp64,
    no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", _LIB, _SRC, "-lm"])
    return _LIB


def _open(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    i = ctypes.c_int
    lib.oracle_round_bf16.argtypes = [ctypes.c_double]
    lib.oracle_round_bf16.restype = ctypes.c_double
    lib.oracle_bin.argtypes = [i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    lib.oracle_head.argtypes = [i, i, i, i, i, i, i, i, i, i, i, dp, dp, dp, i, ip,
                                dp, ip, ip, dp, dp, dp, dp, dp]
    lib.oracle_head.restype = i
    lib.oracle_forward.argtypes = [i, i, i, i, i, i, i, i, i, i, i, i, dp, dp, dp, dp, ip, ip]
    lib.oracle_forward.restype = i
    lib.oracle_backward_head.argtypes = [i, i, i, i, i, i, i, i, i, i, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_backward_head.restype = i
    lib.oracle_pool.argtypes = [i, i, i, i, i, i, dp, dp]
    lib.oracle_pool.restype = None
    lib.oracle_scores.argtypes = [i, i, i, dp, dp, dp]
    lib.oracle_scores.restype = None
    lib.oracle_topk.argtypes = [i, i, i, dp, ip]
    lib.oracle_topk.restype = None
    lib.oracle_landmark_values.argtypes = [i, i, i, i, dp, dp, dp]
    lib.oracle_landmark_values.restype = None
    lib.oracle_route_one.argtypes = [i, i, dp, dp, dp]
    lib.oracle_route_one.restype = i
    lib.oracle_attend_one.argtypes = [i, i, i, i, i, dp, dp, ip, dp, dp, dp, dp, dp]
    lib.oracle_attend_one.restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _open(build())
    return _lib


@contextlib.contextmanager
def swapped_library(path):
    """Run the wrapper against another build of the oracle source (used by
    the tests that plant mistakes in a copy of it)."""
    global _lib
    saved = _lib
    _lib = _open(path)
    try:
        yield
    finally:
        _lib = saved


def _dp(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def round_bf16(x: float) -> float:
    """Nearest bfloat16 value of ``x`` (ties to even)."""
    return _load().oracle_round_bf16(float(x))


def pool_bin(i: int, G: int, P: int) -> tuple[int, int]:
    """Adaptive-average-pooling bin [lo, hi) of output cell ``i`` (G -> P)."""
    lo, hi = ctypes.c_int(), ctypes.c_int()
    _load().oracle_bin(i, G, P, ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact upcast of bf16 / fp32 values
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def head(Q, K, V, grid, m: int, k: int, io: str = "f64", queries=None, debug: bool = False,
         shared: bool = True, s: int = 1):
    """Run the oracle on one head.

    Q, K, V: [N, d] arrays (values are taken exactly; bf16/fp32 torch tensors
    are upcast exactly).  grid = (gh, gw, ph, pw).  ``io`` is the type that
    Q_l, V_l and out are rounded to.  ``queries``: optional list of query
    indices (default all).  Returns a dict with out [nq,d], idx [m,k],
    route [nq] and, with ``debug``, Ql, Vl, R [m,N] (raw scores),
    A [nq,m] (raw query-landmark scores) and W [nq, m+k] (attention weights).
    ``shared=False`` is the routing-only variant: one softmax over the k
    routed logits alone (the shared weights are zero).  ``s > 1`` routes each
    query to its s best landmarks and takes one softmax over the shared
    logits and the union of their experts' keys (W is then not returned;
    route holds the best landmark).
    """
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    N, d = Q.shape
    gh, gw, ph, pw = grid
    qlist = None if queries is None else np.ascontiguousarray(queries, dtype=np.int32)
    nq = N if qlist is None else len(qlist)
    out = np.zeros((nq, d))
    idx = np.zeros((m, k), dtype=np.int32)
    route = np.zeros(nq, dtype=np.int32)
    Ql = np.zeros((m, d)) if debug else None
    Vl = np.zeros((m, d)) if debug else None
    R = np.zeros((m, N)) if debug else None
    A = np.zeros((nq, m)) if debug else None
    W = np.zeros((nq, m + k)) if debug and s == 1 else None
    rc = lib.oracle_head(N, d, gh, gw, ph, pw, m, k, _IO_NAMES[io], int(shared), int(s), _dp(Q), _dp(K), _dp(V),
                         nq, _ip(qlist), _dp(out), _ip(idx), _ip(route),
                         _dp(Ql), _dp(Vl), _dp(R), _dp(A), _dp(W))
    if rc != 0:
        raise ValueError("oracle: invalid sizes")
    res = {"out": out, "idx": idx, "route": route}
    if debug:
        res.update(Ql=Ql, Vl=Vl, R=R, A=A)
        if W is not None:
            res["W"] = W
    return res


def forward(Q, K, V, grid, m: int, k: int, io: str = "f64", shared: bool = True, s: int = 1):
    """Run the oracle on a [B, H, N, d] batch; returns out [B,H,N,d] (fp64,
    holding values of the I/O type), idx [B,H,m,k] and route [B,H,N]."""
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = Q.shape
    gh, gw, ph, pw = grid
    out = np.zeros((B, H, N, d))
    idx = np.zeros((B, H, m, k), dtype=np.int32)
    route = np.zeros((B, H, N), dtype=np.int32)
    rc = lib.oracle_forward(B * H, N, d, gh, gw, ph, pw, m, k, _IO_NAMES[io], int(shared), int(s),
                            _dp(Q), _dp(K), _dp(V), _dp(out), _ip(idx), _ip(route))
    if rc != 0:
        raise ValueError("oracle: invalid sizes")
    return {"out": out, "idx": idx, "route": route}


def backward(Q, K, V, dOut, grid, m: int, k: int, io: str = "f64", shared: bool = True):
    """Gradients dQ, dK, dV [N, d] of one head (s = 1) for the output gradient
    dOut [N, d]; experts and routes are constants, the roundings to the I/O
    type pass gradients through.  fp64."""
    lib = _load()
    Q, K, V, dOut = _f64(Q), _f64(K), _f64(V), _f64(dOut)
    N, d = Q.shape
    gh, gw, ph, pw = grid
    dQ, dK, dV = np.zeros((N, d)), np.zeros((N, d)), np.zeros((N, d))
    rc = lib.oracle_backward_head(N, d, gh, gw, ph, pw, m, k, _IO_NAMES[io], int(shared), _dp(Q), _dp(K), _dp(V),
                                  _dp(dOut), _dp(dQ), _dp(dK), _dp(dV))
    if rc != 0:
        raise ValueError("oracle: invalid sizes")
    return dQ, dK, dV


def attend_one(q, A, expert, K, V, Vl, io: str = "f64", shared: bool = True):
    """Step 6 for one query: one softmax over the m shared logits (raw
    query-landmark scores ``A`` [m], scaled here) and the routed logits of the
    keys listed in ``expert`` (any k key indices), applied to [V_l ; V[expert]].
    The arguments are the oracle's own intermediates (``head(debug=True)``)
    or alternatives the caller builds from them; returns out [d]."""
    lib = _load()
    q, A, K, V, Vl = _f64(q), _f64(A), _f64(K), _f64(V), _f64(Vl)
    E = np.ascontiguousarray(expert, dtype=np.int32)
    d, m, k = q.shape[0], A.shape[0], E.shape[0]
    out = np.zeros(d)
    lib.oracle_attend_one(d, m, k, _IO_NAMES[io], int(shared), _dp(q), _dp(A), _ip(E), _dp(K), _dp(V), _dp(Vl),
                          _dp(out), None)
    return out


def scores_row(Ql_i, K):
    """Raw landmark scores R[i, :] = Q_l[i] . K^T of one landmark (step 2)."""
    lib = _load()
    Ql_i, K = _f64(Ql_i).reshape(1, -1), _f64(K)
    N, d = K.shape
    R = np.zeros(N)
    lib.oracle_scores(N, d, 1, _dp(Ql_i), _dp(K), _dp(R))
    return R


def threads_available() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def head_threaded(Q, K, V, grid, m: int, k: int, io: str = "f64", queries=None, shared: bool = True,
                  threads: int | None = None):
    """The whole operator for one long head, its landmark rows spread over
    host threads (the C routines release the interpreter lock), for the
    queries listed in ``queries`` (default all).  Each landmark row is the
    same sequence of oracle steps as in ``head`` -- scores (2), top-k (3),
    landmark values (4) -- run on that row alone, and each listed query takes
    route (5) and attend (6); no arithmetic differs from ``head``.  Only
    O(N) memory per thread: the raw score rows are not kept (``scores_row``
    recomputes one).  Returns out [nq,d], idx [m,k], route [nq], Ql, Vl,
    A [nq,m] and kth [m], the k-th best raw score of every landmark."""
    from concurrent.futures import ThreadPoolExecutor
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    N, d = Q.shape
    gh, gw, ph, pw = grid
    if gh * gw != N or ph * pw != m or not (1 <= k <= N):
        raise ValueError("oracle: invalid sizes")
    Ql = np.zeros((m, d))
    lib.oracle_pool(gh, gw, ph, pw, d, _IO_NAMES[io], _dp(Q), _dp(Ql))
    idx = np.zeros((m, k), dtype=np.int32)
    Vl = np.zeros((m, d))
    kth = np.zeros(m)

    def landmark(i):
        R = np.zeros(N)
        lib.oracle_scores(N, d, 1, _dp(Ql[i:i + 1]), _dp(K), _dp(R))
        row = np.zeros(k, dtype=np.int32)
        lib.oracle_topk(N, 1, k, _dp(R), _ip(row))
        vl = np.zeros(d)
        lib.oracle_landmark_values(N, d, 1, _IO_NAMES[io], _dp(R), _dp(V), _dp(vl))
        idx[i], Vl[i] = row, vl
        kth[i] = R[row].min()

    with ThreadPoolExecutor(max_workers=threads or threads_available()) as ex:
        list(ex.map(landmark, range(m)))
    qs = np.arange(N) if queries is None else np.asarray(queries)
    out = np.zeros((len(qs), d))
    route = np.zeros(len(qs), dtype=np.int32)
    A = np.zeros((len(qs), m))
    for n, qi in enumerate(qs):
        q = np.ascontiguousarray(Q[qi])
        a = np.zeros(m)
        r = lib.oracle_route_one(d, m, _dp(q), _dp(Ql), _dp(a))
        E = np.ascontiguousarray(idx[r])
        o = np.zeros(d)
        lib.oracle_attend_one(d, m, k, _IO_NAMES[io], int(shared), _dp(q), _dp(a), _ip(E), _dp(K), _dp(V),
                              _dp(Vl), _dp(o), None)
        out[n], route[n], A[n] = o, r, a
    return {"out": out, "idx": idx, "route": route, "Ql": Ql, "Vl": Vl, "A": A, "kth": kth}


def forward_heads_threaded(Q, K, V, grid, m: int, k: int, heads, io: str = "f64", shared: bool = True,
                           s: int = 1, threads: int | None = None):
    """``head`` on each listed (b, h) head of [B, H, N, d] inputs, the heads
    spread over host threads; returns the number of heads run.  Used to time
    the oracle on all host cores."""
    from concurrent.futures import ThreadPoolExecutor
    Qf, Kf, Vf = _f64(Q), _f64(K), _f64(V)

    def one(bh):
        b, h = bh
        head(Qf[b, h], Kf[b, h], Vf[b, h], grid, m, k, io=io, shared=shared, s=s)

    with ThreadPoolExecutor(max_workers=threads or threads_available()) as ex:
        list(ex.map(one, heads))
    return len(heads)
