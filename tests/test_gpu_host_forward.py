"""The forward on host-resident tensors (``mita_forward_host``) through the
C ABI: parity with the CPU oracle on every path, equality with the device
forward's discrete outputs (and, where the kernels do not depend on the
number of heads in a launch, its outputs), chunk ordering across
back-to-back calls, landmarks, pageable memory and argument errors.
"""
import pytest
import torch

import mixture_top_attention_mita_b300 as mita
from mixture_top_attention_mita_b300 import synth
from parity_util import compare_batch

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
PATHS = ["staged", "fused", "tiled"]

SMALL = {
    "tiny_f32": W["tiny_f32"],
    "deit_s": W["deit_s"].scaled(B=3, H=5),          # 15 heads: 8 chunks, the last one short
    "hires56": W["hires56"].scaled(B=1, H=3),
    "long1d_8k": W["long1d"].scaled(B=1, H=2, N=8192, gw=8192, pw=32, m=32),
}


def _plan(w, path="auto", keep=False):
    plan = mita.Plan.for_workload(w)
    plan.set_path(path)
    if keep:
        plan.set_option(mita.OPT_KEEP_LANDMARKS, 1)
    return plan


def _path_ok(w, path):
    plan = _plan(w.scaled(B=1, H=1), path)
    return plan.lib.mita_get_path(plan.handle) >= 0


def _host_outputs(w, pin=True):
    def mk(shape, dtype, fill=None):
        t = torch.empty(shape, dtype=dtype) if fill is None else torch.full(shape, fill, dtype=dtype)
        return t.pin_memory() if pin else t
    io = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return (mk((w.B, w.H, w.N, w.d), io, 0), mk((w.B, w.H, w.m, w.k), torch.int32, -1),
            mk((w.B, w.H, w.N), torch.int32, -1))


def _run_host(plan, w, Q, K, V, pin=True):
    hQ, hK, hV = (t.pin_memory() for t in (Q, K, V)) if pin else (Q, K, V)
    out, idx, route = _host_outputs(w, pin)
    plan.forward_host(hQ, hK, hV, out, idx, route)
    torch.cuda.synchronize()
    assert plan.status() == mita.MITA_OK
    return out, idx, route


def _run_device(w, Q, K, V, path):
    plan = _plan(w, path)
    Qd, Kd, Vd = (t.cuda() for t in (Q, K, V))
    out = torch.empty_like(Qd)
    idx = torch.empty((w.B, w.H, w.m, w.k), dtype=torch.int32, device="cuda")
    route = torch.empty((w.B, w.H, w.N), dtype=torch.int32, device="cuda")
    plan.forward(Qd, Kd, Vd, out, idx, route)
    torch.cuda.synchronize()
    assert plan.status() == mita.MITA_OK
    return out.cpu(), idx.cpu(), route.cpu()


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", sorted(SMALL))
def test_host_forward_matches_oracle_and_device(name, path):
    w = SMALL[name]
    if path != "staged" and not _path_ok(w, path):
        pytest.skip(f"no {path} kernels for this shape")
    Q, K, V = synth.make_inputs(w)
    plan = _plan(w, path)
    out, idx, route = _run_host(plan, w, Q, K, V)
    compare_batch(w, Q, K, V, out, idx, route, exact=False)
    d_out, d_idx, d_route = _run_device(w, Q, K, V, path)
    assert torch.equal(idx, d_idx) and torch.equal(route, d_route)
    if path != "tiled":   # the tiled landmark-value splits depend on the heads per launch
        assert torch.equal(out, d_out)


@pytest.mark.parametrize("path", PATHS)
def test_host_forward_integer_exact(path):
    w = SMALL["deit_s"]
    if path != "staged" and not _path_ok(w, path):
        pytest.skip(f"no {path} kernels for this shape")
    Q, K, V = synth.make_integer_inputs(w)
    out, idx, route = _run_host(_plan(w, path), w, Q, K, V)
    compare_batch(w, Q, K, V, out, idx, route, exact=True)


def test_host_forward_full_size_deit_s_equals_device():
    """The benchmark's DeiT-S layer (1536 heads, 8 chunks of 192)."""
    w = W["deit_s"]
    Q, K, V = synth.make_inputs(w)
    out, idx, route = _run_host(_plan(w), w, Q, K, V)
    d_out, d_idx, d_route = _run_device(w, Q, K, V, "auto")
    assert torch.equal(out, d_out) and torch.equal(idx, d_idx) and torch.equal(route, d_route)


def test_back_to_back_calls_keep_their_own_inputs():
    """Two calls on one stream with no wait between them: the second call's
    chunks reuse the staging slots of the first only after its results left."""
    w = SMALL["deit_s"]
    plan = _plan(w)
    ins = [synth.make_inputs(w, seed=s) for s in (11, 12)]
    pinned = [[t.pin_memory() for t in qkv] for qkv in ins]
    outs = [_host_outputs(w) for _ in ins]
    for (hQ, hK, hV), (o, i, r) in zip(pinned, outs):
        plan.forward_host(hQ, hK, hV, o, i, r)
    torch.cuda.synchronize()
    assert plan.status() == mita.MITA_OK
    for (Q, K, V), (o, i, r) in zip(ins, outs):
        d_out, d_idx, d_route = _run_device(w, Q, K, V, "auto")
        assert torch.equal(o, d_out) and torch.equal(i, d_idx) and torch.equal(r, d_route)


@pytest.mark.parametrize("path", ["fused", "tiled"])
def test_host_forward_landmarks(path):
    w = SMALL["hires56"] if path == "tiled" else SMALL["deit_s"]
    if not _path_ok(w, path):
        pytest.skip(f"no {path} kernels for this shape")
    Q, K, V = synth.make_inputs(w)
    io = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    res = []
    for host in (True, False):
        plan = _plan(w, path, keep=True)
        if host:
            _run_host(plan, w, Q, K, V)
        else:
            Qd, Kd, Vd = (t.cuda() for t in (Q, K, V))
            plan.forward(Qd, Kd, Vd, torch.empty_like(Qd))
        Ql = torch.empty((w.B, w.H, w.m, w.d), dtype=io, device="cuda")
        Vl = torch.empty_like(Ql)
        plan.landmarks(Ql, Vl)
        torch.cuda.synchronize()
        res.append((Ql.cpu(), Vl.cpu()))
    assert torch.equal(res[0][0], res[1][0])
    if path == "fused":
        assert torch.equal(res[0][1], res[1][1])
    else:   # value splits differ with the heads per launch: a few bf16 units at most
        assert torch.allclose(res[0][1].float(), res[1][1].float(), rtol=2e-2, atol=2e-2)


def test_pageable_host_memory():
    w = SMALL["deit_s"]
    Q, K, V = synth.make_inputs(w)
    out, idx, route = _run_host(_plan(w), w, Q, K, V, pin=False)
    d_out, d_idx, d_route = _run_device(w, Q, K, V, "auto")
    assert torch.equal(out, d_out) and torch.equal(idx, d_idx) and torch.equal(route, d_route)


def test_null_optional_outputs_and_launch_count():
    w = SMALL["deit_s"]
    Q, K, V = synth.make_inputs(w)
    plan = _plan(w, "fused")
    hQ, hK, hV = (t.pin_memory() for t in (Q, K, V))
    out = torch.empty_like(Q).pin_memory()
    n0 = plan.launch_count()
    plan.forward_host(hQ, hK, hV, out)
    torch.cuda.synchronize()
    assert plan.status() == mita.MITA_OK
    assert plan.launch_count() - n0 == 8   # one fused launch per chunk (15 heads in chunks of 2)
    d_out, _, _ = _run_device(w, Q, K, V, "fused")
    assert torch.equal(out, d_out)


def test_host_forward_rejects_bad_arguments():
    w = W["deit_t"].scaled(B=1, H=2)
    plan = _plan(w)
    Q = torch.zeros((w.B, w.H, w.N, w.d), dtype=torch.bfloat16)
    with pytest.raises(mita.MitaError) as e:
        plan.forward_host(Q, Q, Q, None)
    assert e.value.code == mita.MITA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        plan.forward_host(Q.cuda(), Q.cuda(), Q.cuda(), Q.cuda())
    s2 = _plan(w, "fused")
    s2.set_option(mita.OPT_ROUTES, 2)
    with pytest.raises(mita.MitaError) as e:
        s2.forward_host(Q, Q, Q, torch.empty_like(Q))
    assert e.value.code == mita.MITA_ERR_UNSUPPORTED
