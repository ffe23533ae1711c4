"""Failure detection on the GPU without a GPU fault.

Bad routing metadata is injected on the host (token ids outside [0, T) written into the routing block
between calls); the kernels must read such rows as zero rows, write nothing for them, report
MOE_ERR_BAD_METADATA in the status block and leave the context usable.  A stuck device wait is made with an
mbarrier that nothing arrives on: the bounded wait must give up with MOE_ERR_DEVICE_TIMEOUT.
"""
import numpy as np
import pytest
import torch

import fine_grained_mixture_gb300 as moe
from fine_grained_mixture_gb300 import synth
from gpu_util import check_routing, run_gpu, to_dev
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_BAD_METADATA = 7


def _routing_still_exact():
    z = torch.randn((300, 16), generator=torch.Generator().manual_seed(5))
    rt, P = moe.moe_route(z.cuda(), 4, "tc", want_P=True)
    check_routing(rt, orc.route(z.numpy(), 4, "tc"), P)


# "pairs" (n = 768): the down-projection and dX~ run on CTA pairs, whose epilogues check the ids the same way
@pytest.mark.parametrize("name,mode", [("tiny", "tc"), ("tiny", "tr"), ("pairs", "tc")])
def test_bad_token_ids_are_flagged_not_followed(name, mode):
    w = synth.custom(700, 256, 768, 6, 2) if name == "pairs" else synth.WORKLOADS["tiny"]
    g = to_dev(synth.make_inputs(w, 0))
    rt = moe.moe_route(g["logits"], w.K, mode)
    torch.cuda.synchronize()
    code, P = rt.device_status()
    assert code == 0 and P > 8
    rt.row_token[3] = -5             # below range
    rt.row_token[7] = w.T + 9        # above range
    O, H = moe.moe_forward(g["X"], g["W1"], g["W2"], rt)
    dX, dW1, dW2, dS = moe.moe_backward(g["dO"], g["X"], g["W1"], g["W2"], H, rt)
    torch.cuda.synchronize()
    code, _ = rt.device_status()
    assert code == MOE_ERR_BAD_METADATA
    for t in (O, H, dX, dW1, dW2, dS):
        assert bool(torch.isfinite(t.float()).all())
    _routing_still_exact()


def test_router_backward_flags_bad_token_ids():
    """The router's row scatter skips rows whose token id is out of range and reports them; the rest of its
    outputs stay finite and the next routing call is exact."""
    w = synth.WORKLOADS["tiny"]
    g = to_dev(synth.make_inputs(w, 1))
    Wr = synth.make_router_weights(w.d, w.E, 1).cuda()
    z = moe.moe_router_forward(g["X"], Wr)
    rt = moe.moe_route(z, w.K, "tc")
    torch.cuda.synchronize()
    assert rt.device_status()[0] == 0
    rt.row_token[0] = -1
    rt.row_token[5] = w.T
    dS = synth.make_row_grads(rt.p_cap, 1).cuda()
    dX = torch.zeros((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    dlogits, dWr = moe.moe_router_backward(dS, rt, z, g["X"], Wr, dX)
    torch.cuda.synchronize()
    assert rt.device_status()[0] == MOE_ERR_BAD_METADATA
    for t in (dlogits, dWr, dX):
        assert bool(torch.isfinite(t.float()).all())
    _routing_still_exact()


def test_stuck_wait_times_out_and_the_context_survives():
    assert moe.selftest_bounded_wait() == MOE_ERR_DEVICE_TIMEOUT
    _routing_still_exact()
    w = synth.WORKLOADS["tiny"]
    out = run_gpu(to_dev(synth.make_inputs(w, 1)), w.K, "tc")
    assert out["code"] == 0
