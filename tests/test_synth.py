"""The seeded input recipe: reproducible, drawn in the documented order with the documented scales, the skewed
workload really leaves experts without tokens, the side generators leave the layer's tensors alone, and the
quantised router inputs make fp32 logits exact in any summation order."""
import math

import numpy as np
import torch

from fine_grained_mixture_gb300 import synth
from oracle import moe_oracle as orc


def test_draws_are_reproducible_and_seeded():
    w = synth.WORKLOADS["tiny"]
    a, b, c = synth.make_inputs(w, 0), synth.make_inputs(w, 0), synth.make_inputs(w, 1)
    for k in a:
        assert torch.equal(a[k], b[k]), k
        assert not torch.equal(a[k], c[k]), k
    assert torch.equal(synth.make_logits_only(w, 0), a["logits"])   # the logits are the first draw


def test_shapes_dtypes_and_scales():
    w = synth.custom(4096, 512, 256, 8, 2)
    g = synth.make_inputs(w, 2)
    assert g["logits"].dtype == torch.float32 and tuple(g["logits"].shape) == (w.T, w.E)
    shapes = dict(X=(w.T, w.d), W1=(w.E, w.d, 2 * w.n), W2=(w.E, w.n, w.d), dO=(w.T, w.d))
    for k, shape in shapes.items():
        assert g[k].dtype == torch.bfloat16 and tuple(g[k].shape) == shape, k
    for k, std in dict(logits=1.0, X=1.0, dO=1.0, W1=1 / math.sqrt(w.d), W2=1 / math.sqrt(w.n)).items():
        t = g[k].double()
        assert abs(t.mean().item()) < 0.02 * std, k
        assert abs(t.std().item() / std - 1) < 0.02, k


def test_skewed_workload_leaves_experts_without_tokens():
    w = synth.WORKLOADS["skew"]
    z = synth.make_logits_only(w, 0).numpy()
    counts = np.bincount(orc.topk_token_choice(z, w.K).ravel(), minlength=w.E)
    assert counts[0] > 0.99 * w.T                 # the largest bias: nearly every token picks expert 0
    assert np.all(np.diff(counts[:16]) < 0)       # popularity falls with the rank of the expert
    assert (counts == 0).sum() > w.E // 4         # many experts get no tokens at all (68 at seed 0)
    plain = synth.make_logits_only(synth.WORKLOADS["fine7b"], 0).numpy()
    assert (np.bincount(orc.topk_token_choice(plain, 8).ravel(), minlength=128) == 0).sum() == 0


def test_side_generators_leave_the_layer_tensors_alone():
    w = synth.WORKLOADS["tiny"]
    before = synth.make_inputs(w, 5)
    u = synth.make_uniforms(w.E, 5)
    Wr = synth.make_router_weights(w.d, w.E, 5)
    dS = synth.make_row_grads(100, 5)
    after = synth.make_inputs(w, 5)
    for k in before:
        assert torch.equal(before[k], after[k]), k
    assert u.min() >= 0 and u.max() < 1 and tuple(u.shape) == (w.E,)
    assert Wr.dtype == torch.bfloat16 and tuple(Wr.shape) == (w.d, w.E) and tuple(dS.shape) == (100,)
    assert torch.equal(u, synth.make_uniforms(w.E, 5)) and not torch.equal(u, synth.make_uniforms(w.E, 6))


def test_quantised_router_inputs_give_exact_fp32_logits():
    gen = torch.Generator().manual_seed(9)
    T, d, E = 64, 2048, 16
    Xq, Wq = synth.quantize_for_exact_logits(torch.randn((T, d), generator=gen).to(torch.bfloat16),
                                             synth.make_router_weights(d, E, 9))
    X, W = Xq.float(), Wq.float()
    assert torch.equal(X * 4, torch.round(X * 4)) and X.abs().max() <= 2
    assert torch.equal(W * 1024, torch.round(W * 1024)) and W.abs().max() <= 0.5
    exact = Xq.double() @ Wq.double()
    prods = X[:, :, None] * W[None, :, :]              # every product exact in fp32
    forward = torch.zeros((T, E))
    backward = torch.zeros((T, E))
    for k in range(d):                                 # two summation orders, one term at a time in fp32
        forward += prods[:, k]
        backward += prods[:, d - 1 - k]
    assert torch.equal(forward.double(), exact) and torch.equal(backward.double(), exact)
    assert torch.equal((X @ W).double(), exact)        # and the library's own blocked order
