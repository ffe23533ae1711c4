"""GPU parity of the router on either side of the layer (through the C ABI) against the CPU oracle.

logits = X W_r: fp32 accumulation of bf16 products, so relative Frobenius error <= 1e-4 (about forty times the
typical fp32 rounding of a d-term dot product) and, on inputs whose logits are exact in fp32 whatever the summation
order, bit-exact.  Router backward: dlogits is computed in fp32 from fp32 inputs (relative error <= 1e-5); dX and
dW_r go through the bf16 copy of dz on the tensor cores and take the layer's bf16 tolerance.
"""
import numpy as np
import pytest
import torch

from fine_grained_mixture_gb300 import synth
from gpu_util import assert_close, f64, run_gpu, to_dev
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu


def _close(name, got, ref, rel_fro, rel_max):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(got - ref).max(initial=0.0) / max(np.abs(ref).max(initial=0.0), 1e-300)
    assert fro <= rel_fro and mx <= rel_max, f"{name}: rel Frobenius {fro:.3e}, rel max {mx:.3e}"


@pytest.mark.parametrize("T,d,E", [(512, 256, 8), (300, 512, 40), (1000, 256, 1024), (24576, 1536, 128)])
def test_router_logits(T, d, E):
    import fine_grained_mixture_gb300 as moe
    gen = torch.Generator().manual_seed(T + d + E)
    X = torch.randn((T, d), generator=gen).to(torch.bfloat16)
    Wr = synth.make_router_weights(d, E, seed=T)
    z = moe.moe_router_forward(X.cuda(), Wr.cuda())
    torch.cuda.synchronize()
    _close("logits", f64(z), orc.router_logits(f64(X), f64(Wr)), 1e-4, 1e-3)


@pytest.mark.parametrize("T,d,E", [(512, 256, 8), (777, 512, 136)])
def test_router_logits_bit_exact_on_exactly_representable_inputs(T, d, E):
    import fine_grained_mixture_gb300 as moe
    gen = torch.Generator().manual_seed(5 * T + E)
    X, Wr = synth.quantize_for_exact_logits(torch.randn((T, d), generator=gen),
                                             synth.make_router_weights(d, E, seed=1) * 8)
    z = moe.moe_router_forward(X.cuda(), Wr.cuda()).cpu().double().numpy()
    assert np.array_equal(z, orc.router_logits(f64(X), f64(Wr)))


def _router_bwd_case(T, d, E, K, mode, seed, dX_in_zero=True):
    import fine_grained_mixture_gb300 as moe
    gen = torch.Generator().manual_seed(seed)
    z = torch.randn((T, E), generator=gen)
    X = torch.randn((T, d), generator=gen).to(torch.bfloat16)
    Wr = synth.make_router_weights(d, E, seed)
    u = synth.make_uniforms(E, seed)
    rt, P = moe.moe_route(z.cuda(), K, mode, want_P=True, uniforms=u.cuda())
    ref = orc.route(z.numpy(), K, mode, u=u.numpy())
    assert P == ref["P"] and np.array_equal(rt.row_token[:P].cpu().numpy(), ref["row_token"])
    dS = synth.make_row_grads(rt.p_cap, seed)
    dX0 = torch.zeros((T, d), dtype=torch.bfloat16) if dX_in_zero else torch.randn((T, d), generator=gen).to(
        torch.bfloat16)
    dX = dX0.cuda()
    dlogits, dWr = moe.moe_router_backward(dS.cuda(), rt, z.cuda(), X.cuda(), Wr.cuda(), dX)
    torch.cuda.synchronize()
    code, _ = rt.device_status()
    assert code == 0
    dz = orc.router_dz(z.numpy(), ref, dS.numpy()[:P].astype(np.float64), mode)
    return dict(dlogits=f64(dlogits), dWr=f64(dWr), dX=f64(dX), dX0=f64(dX0), dz=dz, X=f64(X), Wr=f64(Wr))


@pytest.mark.parametrize("mode", ["tc", "tr", "tr_up", "tr_stoch", "ec"])
@pytest.mark.parametrize("T,d,E,K", [(512, 256, 8, 2), (300, 512, 40, 3), (2048, 256, 256, 8)])
def test_router_backward(T, d, E, K, mode):
    c = _router_bwd_case(T, d, E, K, mode, seed=T + E + K)
    _close("dlogits", c["dlogits"], c["dz"], 1e-5, 1e-5)
    assert_close("dX (router part)", c["dX"], c["dz"] @ c["Wr"].T)
    assert_close("dWr", c["dWr"], c["X"].T @ c["dz"])


def test_router_backward_adds_into_dx():
    c = _router_bwd_case(640, 512, 64, 4, "tc", seed=3, dX_in_zero=False)
    ref = c["dX0"] + c["dz"] @ c["Wr"].T
    assert_close("dX (accumulated)", c["dX"], ref)
    # the router term is visible above the bf16 rounding of dX itself
    assert np.abs(c["dX"] - c["dX0"]).max() > 0


def test_router_backward_full_size_fine7b():
    w = synth.WORKLOADS["fine7b"]
    c = _router_bwd_case(w.T, w.d, w.E, w.K, "tc", seed=0)
    _close("dlogits", c["dlogits"], c["dz"], 1e-5, 1e-5)
    assert_close("dWr", c["dWr"], c["X"].T @ c["dz"])
    rng = np.random.default_rng(0)
    toks = rng.choice(w.T, size=256, replace=False)
    assert_close("dX[sampled tokens]", c["dX"][toks], c["dz"][toks] @ c["Wr"].T)


@pytest.mark.parametrize("mode", ["tc", "tr", "ec"])
def test_router_and_layer_end_to_end(mode):
    """Router forward -> routing -> layer forward/backward -> router backward, against the same chain in the
    oracle.  The inputs make the logits exact in fp32, so both sides route identically."""
    import fine_grained_mixture_gb300 as moe
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, 0)
    Xq, Wr = synth.quantize_for_exact_logits(inp["X"], synth.make_router_weights(w.d, w.E, 0) * 4)
    inp["X"] = Xq
    g = to_dev(inp)
    z = moe.moe_router_forward(g["X"], Wr.cuda())
    g["logits"] = z
    out = run_gpu(g, w.K, mode, uniforms=synth.make_uniforms(w.E, 0))
    assert out["code"] == 0
    dlogits, dWr = moe.moe_router_backward(out["dS"], out["rt"], z, g["X"], Wr.cuda(), out["dX"])
    torch.cuda.synchronize()
    z_ref = orc.router_logits(f64(Xq), f64(Wr))
    assert np.array_equal(f64(z), z_ref)
    rt = orc.route(z_ref.astype(np.float32), w.K, mode)
    P = out["P"]
    assert P == rt["P"] and np.array_equal(out["rt"].row_token[:P].cpu().numpy(), rt["row_token"])
    fwd, bwd = orc.layer(f64(Xq), f64(inp["W1"]), f64(inp["W2"]), f64(inp["dO"]), rt)
    rb = orc.router_backward(z_ref, rt, bwd["dS"], f64(Xq), f64(Wr), mode)
    assert_close("O", f64(out["O"]), fwd["O"])
    assert_close("dlogits", f64(dlogits), rb["dz"])
    assert_close("dX (layer + router)", f64(out["dX"]), bwd["dX"] + rb["dX"])
    assert_close("dWr", f64(dWr), rb["dWr"])
