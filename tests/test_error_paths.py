"""Device-side error reporting, driven from the host with no GPU fault.

A kernel that reads a route outside [0, m) skips it before any access and
sets MITA_ERR_DEVICE; a bounded wait on a barrier that nothing arrives on
gives up and sets MITA_ERR_TIMEOUT.  Both reach the caller through
mita_get_status(), which clears the word, and the plan stays usable."""
import pytest
import torch

import mixture_top_attention_mita_b300 as mita
from mixture_top_attention_mita_b300 import synth

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def _forward_ok(plan, w):
    Q, K, V = (t.cuda() for t in synth.make_inputs(w))
    out = torch.empty_like(Q)
    plan.forward(Q, K, V, out)
    assert plan.status() == mita.MITA_OK
    assert bool(torch.isfinite(out.float()).all())


@pytest.mark.parametrize("name,N", [("deit_t", 196), ("hires56", 3136)])   # warp and block bucket kernels
def test_out_of_range_route_reports_device_error(name, N):
    w = W[name].scaled(B=1, H=2)
    plan = mita.Plan.for_workload(w)
    lib = plan.lib
    route = torch.randint(0, w.m, (w.B, w.H, w.N), dtype=torch.int32, device="cuda")
    assert lib.mita_testing_bucket(plan.handle, route.data_ptr(), None) == mita.MITA_OK
    assert plan.status() == mita.MITA_OK                 # valid routes: nothing reported
    route[0, 1, N // 2] = w.m                            # one landmark past the last
    route[0, 0, 3] = -1
    assert lib.mita_testing_bucket(plan.handle, route.data_ptr(), None) == mita.MITA_OK
    assert plan.status() == mita.MITA_ERR_DEVICE
    assert plan.status() == mita.MITA_OK                 # read once, then cleared
    _forward_ok(plan, w)


def test_bounded_wait_reports_timeout():
    w = W["deit_t"].scaled(B=1, H=1)
    plan = mita.Plan.for_workload(w)
    lib = plan.lib
    assert lib.mita_testing_wait(plan.handle, 0, None) == mita.MITA_ERR_INVALID_ARG
    assert lib.mita_testing_wait(plan.handle, 200000, None) == mita.MITA_OK   # ~0.1 ms of waiting
    assert plan.status() == mita.MITA_ERR_TIMEOUT
    assert plan.status() == mita.MITA_OK
    _forward_ok(plan, w)


def test_status_waits_for_a_side_stream_forward():
    # mita_get_status() waits on the plan's last launch (an event on its
    # stream), so the results are complete once it returns, with no other
    # synchronisation
    w = W["deit_s"].scaled(B=8, H=6)
    Q, K, V = (t.cuda() for t in synth.make_inputs(w))
    plan = mita.Plan.for_workload(w)
    ref = torch.empty_like(Q)
    plan.forward(Q, K, V, ref)
    assert plan.status() == mita.MITA_OK
    side = torch.cuda.Stream()
    out = torch.zeros_like(Q)
    side.wait_stream(torch.cuda.current_stream())
    plan.forward(Q, K, V, out, stream=side)
    assert plan.status() == mita.MITA_OK
    # compared on the current stream, which does not wait for the side stream
    assert bool(torch.equal(out, ref))


def test_workspace_holds_only_what_the_path_needs():
    w = W["deit_s"]
    plan = mita.Plan.for_workload(w)        # the one-kernel path: no score matrix
    fused_bytes = plan.workspace_bytes()
    scores = w.heads * w.m * w.N * 4
    assert fused_bytes < scores
    plan.set_path("staged")                  # the staged path adds the raw scores
    assert plan.workspace_bytes() >= fused_bytes + scores
