"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import fine_grained_mixture_gb300 as moe
from oracle import moe_oracle as orc

# Tolerance of the layer's bf16 tensors with fp32 accumulation (per output and gradient).
REL_FRO = 1e-2
REL_MAX = 3e-2
SCORE_RTOL = 1e-6


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def rel_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mabs = np.abs(got - ref).max(initial=0.0) / max(np.abs(ref).max(initial=0.0), 1e-300)
    return fro, mabs


def assert_close(name, got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if np.abs(ref).max(initial=0.0) == 0.0:
        assert np.abs(got).max(initial=0.0) == 0.0, f"{name}: expected exact zeros"
        return
    fro, mabs = rel_errors(got, ref)
    assert fro <= REL_FRO and mabs <= REL_MAX, f"{name}: rel Frobenius {fro:.3e}, rel max {mabs:.3e}"


def to_dev(inp: dict, dev="cuda") -> dict:
    return {k: v.to(dev) for k, v in inp.items()}


def run_gpu(g: dict, K: int, mode: str, backward=True, uniforms=None, a_from_h=False):
    u = None if uniforms is None else uniforms.to(g["logits"].device)
    rt = moe.moe_route(g["logits"], K, mode, uniforms=u)
    O, H = moe.moe_forward(g["X"], g["W1"], g["W2"], rt, a_from_h=a_from_h)
    out = dict(rt=rt, O=O, H=H)
    if backward:
        dX, dW1, dW2, dS = moe.moe_backward(g["dO"], g["X"], g["W1"], g["W2"], H, rt)
        out.update(dX=dX, dW1=dW1, dW2=dW2, dS=dS)
    torch.cuda.synchronize()
    code, P = rt.device_status()
    out.update(code=code, P=P)
    return out


def check_routing(rt, ref: dict, P: int):
    """Integer metadata bit-exact; scores within SCORE_RTOL."""
    T, K = ref["topk_idx"].shape
    assert P == ref["P"], (P, ref["P"])
    assert np.array_equal(rt.topk_idx.cpu().numpy().reshape(T, K), ref["topk_idx"])
    assert np.array_equal(rt.tc_counts.cpu().numpy(), ref["tc_counts"])
    assert np.array_equal(rt.counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(rt.offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(rt.tile_offsets.cpu().numpy(), ref["tile_offsets"])
    assert np.array_equal(rt.row_token[:P].cpu().numpy(), ref["row_token"])
    assert np.array_equal(rt.row_slot[:P].cpu().numpy(), ref["row_slot"])
    np.testing.assert_allclose(rt.topk_score.cpu().numpy().reshape(T, K), ref["topk_score"], rtol=SCORE_RTOL, atol=0)
    np.testing.assert_allclose(rt.row_score[:P].cpu().numpy(), ref["row_score"], rtol=SCORE_RTOL, atol=0)


def oracle_on_rows(inp: dict, ref: dict, rows: np.ndarray, gpu_scores: np.ndarray | None = None):
    """Oracle forward + backward restricted to `rows` (every output that only depends on them is exact).

    Only the experts the rows touch are converted to fp64; experts are renumbered into that subset."""
    rows = np.asarray(rows, np.int64)
    experts = np.unique(ref["row_expert"][rows])
    remap = {int(e): i for i, e in enumerate(experts)}
    tok = ref["row_token"][rows]
    ex = np.array([remap[int(e)] for e in ref["row_expert"][rows]], dtype=np.int64)
    sc = ref["row_score"][rows] if gpu_scores is None else gpu_scores
    W1 = inp["W1"][torch.from_numpy(experts)].double().numpy()
    W2 = inp["W2"][torch.from_numpy(experts)].double().numpy()
    X = inp["X"].double().numpy()
    dO = inp["dO"].double().numpy() if "dO" in inp else None
    fwd = orc.forward(X, W1, W2, tok, ex, sc)
    bwd = orc.backward(dO, X, W1, W2, tok, ex, sc, fwd) if dO is not None else None
    return experts, fwd, bwd
