"""mita_forward_noalloc: the forward for callers that cannot allocate device
memory (a host framework that owns all device memory through its own pool,
or a latency-critical loop where cudaMalloc would synchronise the device).

It takes its scratch from the library's fixed device array instead of a
plan's workspace.  These checks call it through the C ABI twice in a row and
compare each result with mita_forward() on the same inputs, within the
tolerances the parity tests use.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import mixture_top_attention_mita_b300 as mita
from mixture_top_attention_mita_b300 import synth

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 1e-2), "f32": (1e-5, 1e-5)}


@pytest.mark.parametrize("w", [synth.WORKLOADS["deit_s"].scaled(B=2, H=4), synth.WORKLOADS["tiny_f32"]],
                         ids=["deit_s_small", "tiny_f32"])
def test_noalloc_matches_forward_twice(w):
    dev = torch.device("cuda")
    Q, K, V = (t.to(dev) for t in synth.make_inputs(w))
    plan = mita.Plan.for_workload(w)
    plan.set_path("staged")
    ref_out = torch.empty_like(Q)
    ref_idx = torch.empty(w.B, w.H, w.m, w.k, dtype=torch.int32, device=dev)
    ref_route = torch.empty(w.B, w.H, w.N, dtype=torch.int32, device=dev)
    plan.forward(Q, K, V, ref_out, ref_idx, ref_route)
    assert plan.status() == mita.MITA_OK
    max_tol, mean_tol = TOL[w.dtype]
    out, idx, route = torch.empty_like(Q), torch.empty_like(ref_idx), torch.empty_like(ref_route)
    for call in range(2):
        out.fill_(float("nan"))
        idx.fill_(-1)
        route.fill_(-1)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        mita.forward_noalloc(Q, K, V, out, w.grid, w.m, w.k, idx, route)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if call == 1:   # the first call may load the library's static array
            assert free_before == free_after, "the call allocated device memory"
        diff = (out.double() - ref_out.double()).abs()
        assert torch.isfinite(out.float()).all(), f"call {call}"
        assert float(diff.max()) <= max_tol and float(diff.mean()) <= mean_tol, f"call {call}"
        assert torch.equal(idx, ref_idx) and torch.equal(route, ref_route), f"call {call}"


def test_noalloc_rejects_shapes_beyond_scratch():
    lib = mita.load()
    assert lib.mita_noalloc_scratch_bytes() == 16 * 1024 * 1024
    w = synth.WORKLOADS["deit_s"]   # landmark scores alone need 30 MB
    dev = torch.device("cuda")
    buf = torch.empty(16, dtype=torch.bfloat16, device=dev)
    rc = lib.mita_forward_noalloc(w.B, w.H, w.N, w.d, mita.Grid(*w.grid), w.m, w.k, mita.MITA_BF16,
                                  buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                                  None, None, None)
    assert rc == 2   # MITA_ERR_UNSUPPORTED, before any launch
