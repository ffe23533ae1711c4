"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Routing: bit-exact integer metadata, scores within 1e-6 relative.  Layer tensors (O, H, dX, dW1, dW2, dS):
relative Frobenius error <= 1e-2 and max |err| <= 3e-2 * max |ref| per tensor.  Small shapes compare every
element; the full-size workloads compare sampled tokens, experts and rows that the oracle computes exactly.
"""
import numpy as np
import pytest
import torch

from fine_grained_mixture_gb300 import synth
from gpu_util import (assert_close, check_routing, f64, oracle_on_rows, run_gpu, to_dev)
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

# token choice, token rounding under each rounding rule, expert choice
MODES = ["tc", "tr", "tr_up", "tr_down", "tr_stoch", "ec"]
ROUTE_CASES = [(name, mode) for mode in MODES for name in synth.WORKLOADS]


def _route_both(z, K, mode, seed=0):
    """GPU routing through the C ABI and the oracle's, on the same logits (and uniforms for tr_stoch)."""
    import fine_grained_mixture_gb300 as moe
    u = synth.make_uniforms(z.shape[1], seed)
    rt, P = moe.moe_route(z.cuda(), K, mode, want_P=True, uniforms=u.cuda())
    return rt, P, orc.route(z.numpy(), K, mode, u=u.numpy())


@pytest.mark.parametrize("name,mode", ROUTE_CASES)
def test_routing_workloads(name, mode):
    w = synth.WORKLOADS[name]
    z = synth.make_logits_only(w, 0)
    rt, P, ref = _route_both(z, w.K, mode)
    code, P2 = rt.device_status()
    assert code == 0 and P2 == P
    check_routing(rt, ref, P)


EDGE_SHAPES = [(2048, 1024, 32, False), (1, 8, 2, False), (777, 33, 5, True), (300, 1, 1, False), (4099, 64, 8, True),
               (200, 256, 1, False)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,E,K,ties", EDGE_SHAPES)
def test_routing_edge_shapes(T, E, K, ties, mode):
    gen = torch.Generator().manual_seed(T * 7 + E)
    z = torch.randn((T, E), generator=gen)
    if ties:
        z = torch.round(z * 2) / 2          # many equal logits, -0.0 beside +0.0: every tie-break rule
    rt, P, ref = _route_both(z, K, mode, seed=T)
    check_routing(rt, ref, P)


@pytest.mark.parametrize("T,E,K,modes", [(49152, 128, 8, MODES), (49152, 1024, 32, ["tr", "ec"])])
def test_routing_at_the_largest_token_count(T, E, K, modes):
    """The selection modes keep one expert's keys for all T tokens in shared memory, so T = 49152 is the largest
    count they accept; at that size (and with E and K at their maxima) the metadata is still bit-exact."""
    z = torch.randn((T, E), generator=torch.Generator().manual_seed(T + E))
    for mode in modes:
        rt, P, ref = _route_both(z, K, mode, seed=T)
        check_routing(rt, ref, P)


def test_stochastic_rounding_without_uniforms_is_rejected():
    import fine_grained_mixture_gb300 as moe
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route(torch.randn((64, 8)).cuda(), 2, "tr_stoch")
    assert ei.value.code == 1


def test_routing_nonfinite_logits_flagged():
    import fine_grained_mixture_gb300 as moe
    z = torch.randn((64, 8))
    z[5, 3] = float("nan")
    rt = moe.moe_route(z.cuda(), 2, "tc")
    code, _ = rt.device_status()
    assert code == 5  # MOE_ERR_NONFINITE_LOGITS


def _full_compare(inp, K, mode, a_from_h=False):
    g = to_dev(inp)
    u = synth.make_uniforms(inp["logits"].shape[1], 0)
    out = run_gpu(g, K, mode, uniforms=u, a_from_h=a_from_h)
    assert out["code"] == 0
    ref = orc.route(inp["logits"].numpy(), K, mode, u=u.numpy())
    check_routing(out["rt"], ref, out["P"])
    X, W1, W2, dO = (f64(inp[k]) for k in ("X", "W1", "W2", "dO"))
    fwd, bwd = orc.layer(X, W1, W2, dO, ref)
    P = out["P"]
    assert_close("O", f64(out["O"]), fwd["O"])
    assert_close("H", f64(out["H"][:P]), fwd["H"])
    assert_close("dS", f64(out["dS"][:P]), bwd["dS"])
    assert_close("dX", f64(out["dX"]), bwd["dX"])
    assert_close("dW1", f64(out["dW1"]), bwd["dW1"])
    assert_close("dW2", f64(out["dW2"]), bwd["dW2"])
    empty = np.nonzero(ref["counts"] == 0)[0]
    if len(empty):
        assert float(out["dW1"][torch.from_numpy(empty).cuda()].abs().max()) == 0.0
        assert float(out["dW2"][torch.from_numpy(empty).cuda()].abs().max()) == 0.0


@pytest.mark.parametrize("mode", MODES)
def test_layer_tiny_full(mode):
    w = synth.WORKLOADS["tiny"]
    _full_compare(synth.make_inputs(w, 0), w.K, mode)


@pytest.mark.parametrize("T,d,n,E,K,skew,mode", [
    (300, 256, 128, 5, 2, False, "tc"),      # ragged tail tiles, T not a multiple of 128
    (300, 256, 128, 5, 2, False, "tr"),
    (1000, 512, 256, 16, 4, True, "tc"),     # skewed: experts without tokens, one crowded expert
    (1000, 512, 256, 16, 4, True, "tr"),
    (1, 256, 128, 4, 2, False, "tc"),        # a single token
    (260, 256, 384, 1, 1, False, "tc"),      # one expert holds every token; n = 3 x 128
    (640, 768, 128, 3, 3, False, "tc"),      # K = E: every token visits every expert
    (1000, 512, 256, 16, 4, True, "tr_up"),  # skewed, every expert padded up
    (1000, 512, 256, 16, 4, True, "ec"),     # expert choice: equal counts whatever the skew
    (300, 256, 128, 5, 2, False, "tr_stoch"),
    (100, 256, 128, 64, 1, False, "ec"),     # T K < E: C = 1 row per expert
    # K loops of 768 and more run the scatter-add GEMMs on CTA pairs: experts with odd m-tile counts (a pair's
    # second m-tile past the expert), empty experts, ragged tails
    (700, 256, 768, 6, 2, True, "tc"),
    (300, 512, 1024, 3, 2, False, "tr"),
    (513, 256, 768, 4, 3, False, "ec"),
])
def test_layer_small_shapes(T, d, n, E, K, skew, mode):
    w = synth.custom(T, d, n, E, K, skew=skew)
    _full_compare(synth.make_inputs(w, 1), K, mode)


# The forward that recomputes A = SwiGLU(H) inside the down-projection (A never written): every element at the
# tiny size and on the ragged and skewed shapes, sampled outputs at the four full-size workloads below.
@pytest.mark.parametrize("mode", ["tc", "tr", "ec"])
def test_layer_tiny_full_a_from_h(mode):
    w = synth.WORKLOADS["tiny"]
    _full_compare(synth.make_inputs(w, 0), w.K, mode, a_from_h=True)


@pytest.mark.parametrize("T,d,n,E,K,skew,mode", [
    (300, 256, 128, 5, 2, False, "tc"),      # ragged tail tiles: the producers stop at the expert's last row
    (1000, 512, 256, 16, 4, True, "tr"),     # skewed, empty experts
    (260, 256, 384, 1, 1, False, "tc"),      # n = 3 x 128: the k-blocks of A span the gate and up halves of H
    (1, 256, 128, 4, 2, False, "tc"),        # a single token
])
def test_layer_small_shapes_a_from_h(T, d, n, E, K, skew, mode):
    w = synth.custom(T, d, n, E, K, skew=skew)
    _full_compare(synth.make_inputs(w, 1), K, mode, a_from_h=True)


@pytest.mark.parametrize("name,mode,a_from_h", [
    ("fine7b", "tc", False), ("fine7b", "tr", False), ("coarse", "tc", False), ("sparse", "tc", False),
    ("sparse", "tr", False), ("skew", "tc", False), ("skew", "tr", False), ("sparse", "tr_stoch", False),
    ("skew", "ec", False),
    ("fine7b", "tc", True), ("coarse", "tc", True), ("sparse", "tr", True), ("skew", "tc", True)])
def test_layer_full_size_sampled(name, mode, a_from_h):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, 0)
    g = to_dev(inp)
    u = synth.make_uniforms(w.E, 0)
    out = run_gpu(g, w.K, mode, uniforms=u, a_from_h=a_from_h)
    assert out["code"] == 0
    ref = orc.route(inp["logits"].numpy(), w.K, mode, u=u.numpy())
    check_routing(out["rt"], ref, out["P"])
    rng = np.random.default_rng(0)
    # tokens: O and dX of sampled tokens need exactly the rows of those tokens
    toks = rng.choice(w.T, size=48, replace=False)
    rows = np.nonzero(np.isin(ref["row_token"], toks))[0]
    _, fwd, bwd = oracle_on_rows(inp, ref, rows)
    tsel = torch.from_numpy(toks)
    O_ref = fwd["O"][toks]
    dX_ref = bwd["dX"][toks]
    assert_close("O[sampled tokens]", f64(out["O"].cpu()[tsel]), O_ref)
    assert_close("dX[sampled tokens]", f64(out["dX"].cpu()[tsel]), dX_ref)
    rsel = torch.from_numpy(rows)
    assert_close("H[rows of sampled tokens]", f64(out["H"].cpu()[rsel]), fwd["H"])
    assert_close("dS[rows of sampled tokens]", f64(out["dS"].cpu()[rsel]), bwd["dS"])
    # experts: the largest and a median non-empty one; empty experts must give exact zeros
    counts = ref["counts"]
    live = np.nonzero(counts > 0)[0]
    picks = [int(np.argmax(counts)), int(live[np.argsort(counts[live])[len(live) // 2]])]
    for e in picks:
        erows = np.arange(ref["offsets"][e], ref["offsets"][e + 1])
        _, fe, be = oracle_on_rows(inp, ref, erows)
        assert_close(f"dW1[{e}]", f64(out["dW1"][e]), be["dW1"][0])
        assert_close(f"dW2[{e}]", f64(out["dW2"][e]), be["dW2"][0])
    for e in np.nonzero(counts == 0)[0][:4]:
        assert float(out["dW1"][int(e)].abs().max()) == 0.0
        assert float(out["dW2"][int(e)].abs().max()) == 0.0
