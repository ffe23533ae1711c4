"""The layer inside a CUDA graph.

Every call forks its memory-bound side work (accumulator zeroing, the dX cast) onto a library-owned stream
and joins it back with events, and launches its kernels with programmatic dependent launch.  Captured on a
caller stream and replayed, route + forward + backward must give the eager results: routing bit-exact, the
fp32-accumulated tensors within the parity tolerance (their reduce-add order may differ run to run).
"""
import pytest
import torch

import fine_grained_mixture_gb300 as moe
from fine_grained_mixture_gb300 import synth
from gpu_util import assert_close, f64, to_dev

pytestmark = pytest.mark.gpu


# token rounding runs its fill as clusters of 8 (tiny), 4 (fine7b) and 2 (sparse) CTAs per expert; the sparse
# layer's weight gradients take the merged 256-row launch; a_from_h: the down-projection recomputes A from H;
# "pairs" (n = 768): the down-projection and dX~ run on CTA pairs (two-CTA clusters)
PAIRS = synth.custom(700, 256, 768, 6, 2, skew=True)


@pytest.mark.parametrize("name,mode,a_from_h", [("tiny", "tc", False), ("tiny", "tr", False), ("fine7b", "tc", False),
                                               ("fine7b", "tr", True), ("sparse", "tr", False), ("pairs", "tc", False),
                                               ("pairs", "tr", False)])
def test_route_forward_backward_replay_in_a_cuda_graph(name, mode, a_from_h):
    w = PAIRS if name == "pairs" else synth.WORKLOADS[name]
    g = to_dev(synth.make_inputs(w, 3))
    rt = moe.Routing(w.T, w.E, w.K, mode, "cuda")
    p = rt.p_cap
    bf = torch.bfloat16
    O = torch.empty((w.T, w.d), dtype=bf, device="cuda")
    H = torch.empty((p, 2 * w.n), dtype=bf, device="cuda")
    dX = torch.empty((w.T, w.d), dtype=bf, device="cuda")
    dW1 = torch.empty((w.E, w.d, 2 * w.n), dtype=bf, device="cuda")
    dW2 = torch.empty((w.E, w.n, w.d), dtype=bf, device="cuda")
    dS = torch.empty(p, dtype=torch.float32, device="cuda")
    fflags = moe.MOE_FLAG_A_FROM_H if a_from_h else 0
    wsf = torch.empty(moe.moe_forward_workspace_size(w.T, w.d, w.n, w.E, w.K, p, fflags), dtype=torch.uint8,
                      device="cuda")
    wsb = torch.empty(moe.moe_backward_workspace_size(w.T, w.d, w.n, w.E, w.K, p), dtype=torch.uint8, device="cuda")

    def step():
        moe.moe_route(g["logits"], w.K, mode, routing=rt)
        moe.moe_forward(g["X"], g["W1"], g["W2"], rt, O=O, H=H, ws=wsf, a_from_h=a_from_h)
        moe.moe_backward(g["dO"], g["X"], g["W1"], g["W2"], H, rt, dX=dX, dW1=dW1, dW2=dW2, dS=dS, ws=wsb)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager: first-use set-up (attributes, side stream, events) happens outside the capture
    torch.cuda.synchronize()
    eager = {k: t.clone() for k, t in dict(O=O, H=H, dX=dX, dW1=dW1, dW2=dW2, dS=dS, row_token=rt.row_token,
                                             offsets=rt.offsets).items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for t in (O, H, dX, dW1, dW2, dS):
        t.zero_()
    rt.row_token.fill_(-1)
    torch.cuda.synchronize()
    graph.replay()
    graph.replay()  # twice: nothing from the first replay may leak into the second
    torch.cuda.synchronize()
    code, P = rt.device_status()
    assert code == 0
    assert torch.equal(rt.offsets, eager["offsets"])
    assert torch.equal(rt.row_token[:P], eager["row_token"][:P])
    for k, t in dict(O=O, H=H[:P], dX=dX, dW1=dW1, dW2=dW2, dS=dS[:P]).items():
        ref = eager[k][:P] if k in ("H", "dS") else eager[k]
        assert_close(k, f64(t), f64(ref))


@pytest.mark.parametrize("mode", ["tr", "ec"])
def test_router_and_deterministic_layer_replay_bitwise(mode):
    """Router forward, routing, the deterministic forward and backward, and the router backward in one CUDA graph:
    with fixed-point aggregation and the router's fixed-order sums every output is reproducible, so each replay
    must equal the eager run bit for bit."""
    w = synth.WORKLOADS["tiny"]
    g = to_dev(synth.make_inputs(w, 4))
    Wr = synth.make_router_weights(w.d, w.E, 4).cuda()
    rt = moe.Routing(w.T, w.E, w.K, mode, "cuda")
    p = rt.p_cap
    bf = torch.bfloat16
    flags = moe.MOE_FLAG_DETERMINISTIC
    z = torch.empty((w.T, w.E), dtype=torch.float32, device="cuda")
    O = torch.empty((w.T, w.d), dtype=bf, device="cuda")
    H = torch.empty((p, 2 * w.n), dtype=bf, device="cuda")
    dX = torch.empty((w.T, w.d), dtype=bf, device="cuda")
    dW1 = torch.empty((w.E, w.d, 2 * w.n), dtype=bf, device="cuda")
    dW2 = torch.empty((w.E, w.n, w.d), dtype=bf, device="cuda")
    dS = torch.empty(p, dtype=torch.float32, device="cuda")
    dz = torch.empty((w.T, w.E), dtype=torch.float32, device="cuda")
    dWr = torch.empty((w.d, w.E), dtype=torch.float32, device="cuda")
    wsf = torch.empty(moe.moe_forward_workspace_size(w.T, w.d, w.n, w.E, w.K, p, flags), dtype=torch.uint8,
                      device="cuda")
    wsb = torch.empty(moe.moe_backward_workspace_size(w.T, w.d, w.n, w.E, w.K, p, flags), dtype=torch.uint8,
                      device="cuda")

    def step():
        moe.moe_router_forward(g["X"], Wr, logits=z)
        moe.moe_route(z, w.K, mode, routing=rt)
        moe.moe_forward(g["X"], g["W1"], g["W2"], rt, O=O, H=H, ws=wsf, deterministic=True)
        moe.moe_backward(g["dO"], g["X"], g["W1"], g["W2"], H, rt, dX=dX, dW1=dW1, dW2=dW2, dS=dS, ws=wsb,
                         deterministic=True)
        moe.moe_router_backward(dS, rt, z, g["X"], Wr, dX, dlogits=dz, dWr=dWr)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager: first-use set-up happens outside the capture
    torch.cuda.synchronize()
    code, P = rt.device_status()
    assert code == 0
    outs = dict(z=z, O=O, dX=dX, dW1=dW1, dW2=dW2, dz=dz)
    eager = {k: t.clone() for k, t in outs.items()}
    eager.update(H=H[:P].clone(), dS=dS[:P].clone(), dWr=dWr.clone())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for _ in range(2):
        for t in list(outs.values()) + [H, dS, dWr]:
            t.zero_()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert rt.device_status() == (0, P)
        for k, t in outs.items():
            assert torch.equal(t, eager[k]), k
        assert torch.equal(H[:P], eager["H"]) and torch.equal(dS[:P], eager["dS"])
        assert torch.equal(dWr, eager["dWr"])
