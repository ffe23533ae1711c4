"""Seeded synthetic inputs for the MoE expert layer (shared by the tests, the bench and the oracle runs).

This module holds no part of the layer's arithmetic: it only draws router logits, activations, weights
and the upstream gradient with a fixed recipe, so that the CUDA path and the CPU oracle see the very
same host tensors.

Recipe (per workload, one ``torch.Generator('cpu')`` seeded with ``seed``), drawn in this order:

* ``logits`` fp32 [T, E] ~ N(0, 1); the skewed workload adds a per-expert bias
  b_e = 2 * ln(1 / rank_e) with rank_e = e + 1, so expert popularity is Zipf-like;
* ``X``  [T, d] ~ N(0, 1), rounded to bf16 (round to nearest even);
* ``W1`` [E, d, 2n] ~ N(0, 1/d), drawn one expert at a time, bf16; columns [0, n) are the gate
  projection and [n, 2n) the up projection;
* ``W2`` [E, n, d] ~ N(0, 1/n), drawn one expert at a time, bf16;
* ``dO`` [T, d] ~ N(0, 1), bf16.

The router weights W_r [d, E] ~ N(0, 1/d) (bf16) and synthetic per-row gradients dS come from generators of their
own as well.  Stochastic rounding draws one uniform per expert; ``make_uniforms`` takes them from a generator of their own
(seeded with ``seed + 0x5EED``) so the tensors above are the same whichever routing mode is run.

The workloads are the layer shapes SonicMoE is evaluated on in spirit (a fine-grained 7B-class layer,
a coarser layer, a high-sparsity layer and a skewed-load layer); the pages list no public dataset,
so these seeded draws stand in for real activations.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

M_TILE = 128


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    n: int
    E: int
    K: int
    skew: bool = False

    @property
    def dims(self):
        return dict(T=self.T, d=self.d, n=self.n, E=self.E, K=self.K)


WORKLOADS = {
    "tiny": Workload("tiny", T=512, d=256, n=128, E=8, K=2),
    "fine7b": Workload("fine7b", T=24576, d=1536, n=256, E=128, K=8),
    "coarse": Workload("coarse", T=16384, d=4096, n=1024, E=128, K=8),
    "sparse": Workload("sparse", T=16384, d=1536, n=256, E=256, K=4),
    "skew": Workload("skew", T=32768, d=2048, n=768, E=128, K=8, skew=True),
}


def custom(T, d, n, E, K, skew=False, name="custom") -> Workload:
    return Workload(name, T=T, d=d, n=n, E=E, K=K, skew=skew)


def make_logits(w: Workload, gen: torch.Generator) -> torch.Tensor:
    z = torch.randn((w.T, w.E), generator=gen, dtype=torch.float32)
    if w.skew:
        bias = torch.tensor([2.0 * math.log(1.0 / (e + 1)) for e in range(w.E)], dtype=torch.float32)
        z = z + bias[None, :]
    return z.contiguous()


def make_inputs(w: Workload, seed: int = 0, with_grad: bool = True) -> dict:
    """Draw the workload's tensors on the host (CPU), in the documented order."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    logits = make_logits(w, gen)
    X = torch.randn((w.T, w.d), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    W1 = torch.empty((w.E, w.d, 2 * w.n), dtype=torch.bfloat16)
    s1 = 1.0 / math.sqrt(w.d)
    for e in range(w.E):
        W1[e] = (torch.randn((w.d, 2 * w.n), generator=gen, dtype=torch.float32) * s1).to(torch.bfloat16)
    W2 = torch.empty((w.E, w.n, w.d), dtype=torch.bfloat16)
    s2 = 1.0 / math.sqrt(w.n)
    for e in range(w.E):
        W2[e] = (torch.randn((w.n, w.d), generator=gen, dtype=torch.float32) * s2).to(torch.bfloat16)
    out = dict(logits=logits, X=X, W1=W1, W2=W2)
    if with_grad:
        out["dO"] = torch.randn((w.T, w.d), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_logits_only(w: Workload, seed: int = 0) -> torch.Tensor:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return make_logits(w, gen)


def make_uniforms(E: int, seed: int = 0) -> torch.Tensor:
    """Per-expert uniforms in [0, 1) for stochastic rounding (fp32, host)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 0x5EED)
    return torch.rand((E,), generator=gen, dtype=torch.float32)


def make_router_weights(d: int, E: int, seed: int = 0) -> torch.Tensor:
    """Router weights W_r [d, E] ~ N(0, 1/d), bf16, from a generator of their own (seed + 0x2047)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 0x2047)
    return (torch.randn((d, E), generator=gen, dtype=torch.float32) / math.sqrt(d)).to(torch.bfloat16)


def make_row_grads(P: int, seed: int = 0) -> torch.Tensor:
    """Per-row upstream gradients dS [P] ~ N(0, 1), fp32, from a generator of their own (seed + 0xD5)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 0xD5)
    return torch.randn((P,), generator=gen, dtype=torch.float32)


def quantize_for_exact_logits(X: torch.Tensor, Wr: torch.Tensor):
    """X on a grid of 1/4 in [-2, 2] and W_r on a grid of 2^-10 in [-1/2, 1/2] (both stay on their grids in bf16):
    every product of z = X W_r is a multiple of 2^-12 and, for d <= 2048, every partial sum stays below 2^12 in
    magnitude, so fp32 accumulation in any order gives z exactly and the routing cannot depend on the order."""
    Xq = torch.clamp(torch.round(X.float() * 4) / 4, -2, 2).to(torch.bfloat16)
    Wq = torch.clamp(torch.round(Wr.float() * 1024) / 1024, -0.5, 0.5).to(torch.bfloat16)
    return Xq, Wq
