"""Token-sharded data parallelism of the MoE expert layer: one process per GPU, each with a full replica of the
expert weights W1 [E, d, 2n] and W2 [E, n, d] and its own shard of the batch's tokens.

SonicMoE trains with plain data parallelism (FSDP-2 over the GPUs; arXiv abstract, and the reading note's
"Experiments / main results"): every GPU routes and runs the layer on its own tokens, and the only exchange the
layer needs is the sum of the weight gradients over the GPUs.  Nothing else crosses ranks:

* token-choice routing is decided per token (a token's top-K of its own logits), so a shard routes exactly as the
  same tokens would inside the whole batch, and O, H, dX and dS of a token depend only on that token's rows;
* dW1_e = sum over the rows of expert e of X_t^T dH_r and dW2_e = sum of (sA_r)^T dO_t are sums over tokens, so the
  sum over ranks of each rank's dW over its shard equals dW over the whole batch.

Token rounding and expert choice rank each expert's candidates among the tokens a rank holds, so under data
parallelism they round each rank's per-expert counts to multiples of M_tile (as a data-parallel trainer that routes
each micro-batch on its own GPU does); their results are per-shard, not those of one batch of all tokens.

This module holds the host side only: the shard bounds and the all-reduce over ``torch.distributed`` (NCCL
between GPUs, gloo on the CPU).  The layer itself runs in libmoe on each rank.
"""
from __future__ import annotations

import os

import torch


def token_shard(T: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of rank's contiguous share of T tokens; shares differ by at most one token and tile [0, T)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if T < 0:
        raise ValueError(f"negative token count {T}")
    return rank * T // world, (rank + 1) * T // world


def allreduce_weight_grads(dW1: torch.Tensor, dW2: torch.Tensor, group=None, async_op: bool = False):
    """Sums dW1 and dW2 over the ranks of `group`, in place (one all-reduce each, in that order).

    Returns the two work handles when async_op (the caller waits on them before using the gradients), else
    None.  With a single rank (or no process group) nothing is exchanged."""
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return [] if async_op else None
    works = [dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group, async_op=async_op) for t in (dW1, dW2)]
    return works if async_op else None


def broadcast_weights(W1: torch.Tensor, W2: torch.Tensor, src: int = 0, group=None) -> None:
    """Makes every rank's replica equal to rank `src`'s (the data-parallel start state)."""
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return
    for t in (W1, W2):
        dist.broadcast(t, src=src, group=group)


def nccl_environment() -> None:
    """Settings for the NCCL process group of the layer's replicas: NVLink SHARP (NVLS) multicast stays off, so
    the all-reduce runs on plain peer copies and no GPU memory is bound to a multicast object."""
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
