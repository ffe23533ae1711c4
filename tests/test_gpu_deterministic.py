"""Deterministic aggregation (MOE_FLAG_DETERMINISTIC) through the C ABI: the same parity bar as the default path
against the CPU oracle, and bitwise-identical outputs on repeated runs (fixed-point sums do not depend on the
order in which the GPU lands the rows' contributions)."""
import numpy as np
import pytest
import torch

import fine_grained_mixture_gb300 as moe
from fine_grained_mixture_gb300 import synth
from gpu_util import assert_close, check_routing, f64, oracle_on_rows, to_dev
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu


def _run(g, K, mode, det=True, W2=None):
    rt = moe.moe_route(g["logits"], K, mode)
    O, H = moe.moe_forward(g["X"], g["W1"], g["W2"] if W2 is None else W2, rt, deterministic=det)
    dX, dW1, dW2, dS = moe.moe_backward(g["dO"], g["X"], g["W1"], g["W2"] if W2 is None else W2, H, rt,
                                        deterministic=det)
    torch.cuda.synchronize()
    code, P = rt.device_status()
    return dict(rt=rt, O=O, H=H[:P], dX=dX, dW1=dW1, dW2=dW2, dS=dS[:P], code=code, P=P)


@pytest.mark.parametrize("T,d,n,E,K,mode", [(512, 256, 128, 8, 2, "tc"), (512, 256, 128, 8, 2, "tr"),
                                            (1000, 512, 512, 16, 4, "tc"), (300, 256, 384, 5, 2, "ec"),
                                            (400, 256, 768, 5, 2, "tc")])   # CTA-pair down-projection and dX~
def test_deterministic_matches_oracle(T, d, n, E, K, mode):
    w = synth.custom(T, d, n, E, K)
    inp = synth.make_inputs(w, 2)
    out = _run(to_dev(inp), K, mode)
    assert out["code"] == 0
    ref = orc.route(inp["logits"].numpy(), K, mode)
    check_routing(out["rt"], ref, out["P"])
    fwd, bwd = orc.layer(f64(inp["X"]), f64(inp["W1"]), f64(inp["W2"]), f64(inp["dO"]), ref)
    for name, r in (("O", fwd["O"]), ("H", fwd["H"]), ("dX", bwd["dX"]), ("dW1", bwd["dW1"]), ("dW2", bwd["dW2"]),
                    ("dS", bwd["dS"])):
        assert_close(name, f64(out[name]), r)


@pytest.mark.parametrize("name,T,d,n,E,K", [("n512", 4096, 512, 512, 32, 4), ("fine7b", 24576, 1536, 256, 128, 8)])
def test_deterministic_is_bitwise_reproducible(name, T, d, n, E, K):
    w = synth.WORKLOADS["fine7b"] if name == "fine7b" else synth.custom(T, d, n, E, K)
    g = to_dev(synth.make_inputs(w, 0))
    a = _run(g, K, "tc")
    b = _run(g, K, "tc")
    assert a["code"] == 0 and b["code"] == 0
    for key in ("O", "H", "dX", "dW1", "dW2", "dS"):
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key].view(torch.int32),
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key].view(torch.int32)), key
    # and the default (fp32 atomic) path agrees with it within the layer's tolerance
    c = _run(g, K, "tc", det=False)
    for key in ("O", "dX", "dS"):
        assert_close(key, f64(c[key]), f64(a[key]).astype(np.float64))


def test_deterministic_range_overflow_is_reported():
    w = synth.WORKLOADS["tiny"]
    g = to_dev(synth.make_inputs(w, 0))
    big = (g["W2"].float() * 1e8).to(torch.bfloat16)   # contributions far beyond 2^21
    out = _run(g, w.K, "tc", W2=big)
    assert out["code"] == 9  # MOE_ERR_RANGE
    ok = _run(g, w.K, "tc")  # the next call on normal data is clean again
    assert ok["code"] == 0


def test_deterministic_full_size_matches_oracle_on_samples():
    """At the fine7b size the deterministic path is checked against the oracle itself, not only against the default
    path: O, dX and dS of sampled tokens (which need exactly those tokens' rows), H of those rows, and dW1/dW2 of
    the largest and a median expert."""
    w = synth.WORKLOADS["fine7b"]
    inp = synth.make_inputs(w, 0)
    out = _run(to_dev(inp), w.K, "tc")
    assert out["code"] == 0
    ref = orc.route(inp["logits"].numpy(), w.K, "tc")
    check_routing(out["rt"], ref, out["P"])
    rng = np.random.default_rng(1)
    toks = rng.choice(w.T, size=48, replace=False)
    rows = np.nonzero(np.isin(ref["row_token"], toks))[0]
    _, fwd, bwd = oracle_on_rows(inp, ref, rows)
    tsel, rsel = torch.from_numpy(toks), torch.from_numpy(rows)
    assert_close("O[sampled tokens]", f64(out["O"].cpu()[tsel]), fwd["O"][toks])
    assert_close("dX[sampled tokens]", f64(out["dX"].cpu()[tsel]), bwd["dX"][toks])
    assert_close("H[rows of sampled tokens]", f64(out["H"].cpu()[rsel]), fwd["H"])
    assert_close("dS[rows of sampled tokens]", f64(out["dS"].cpu()[rsel]), bwd["dS"])
    counts = ref["counts"]
    live = np.nonzero(counts > 0)[0]
    for e in (int(np.argmax(counts)), int(live[np.argsort(counts[live])[len(live) // 2]])):
        _, _, be = oracle_on_rows(inp, ref, np.arange(ref["offsets"][e], ref["offsets"][e + 1]))
        assert_close(f"dW1[{e}]", f64(out["dW1"][e]), be["dW1"][0])
        assert_close(f"dW2[{e}]", f64(out["dW2"][e]), be["dW2"][0])


@pytest.mark.parametrize("mode", ["tc", "tr"])
def test_deterministic_with_a_kept_off_hbm(mode):
    """Both forward flags at once: the down-projection that recomputes A from H, with the fixed-point aggregation.
    Against the oracle, and bitwise identical on a second run."""
    w = synth.custom(300, 256, 384, 5, 2)   # ragged tail tiles; n = 3 x 128
    inp = synth.make_inputs(w, 3)
    g = to_dev(inp)
    outs = []
    for _ in range(2):
        rt = moe.moe_route(g["logits"], w.K, mode)
        O, H = moe.moe_forward(g["X"], g["W1"], g["W2"], rt, deterministic=True, a_from_h=True)
        torch.cuda.synchronize()
        code, P = rt.device_status()
        assert code == 0
        outs.append((O.clone(), H[:P].clone(), P))
    ref = orc.route(inp["logits"].numpy(), w.K, mode)
    fwd, _ = orc.layer(f64(inp["X"]), f64(inp["W1"]), f64(inp["W2"]), f64(inp["dO"]), ref)
    assert_close("O", f64(outs[0][0]), fwd["O"])
    assert_close("H", f64(outs[0][1]), fwd["H"])
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
