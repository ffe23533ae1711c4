"""What the forward leaves on the device for the backward.

The method keeps only X, H and the routing metadata between forward and backward: 2Td + 4TKn bytes for token
choice, plus the metadata ("SonicMoE: Accelerating MoE with IO and Tile-aware Optimizations" reading note,
"Key design 3: minimal-activation-cache backward"; H is the [P, 2n] pre-activation).  Measured here as the
caching allocator's growth across route + forward, after the output O is released: the forward's transient
workspace (A and the fp32 accumulator) must be gone, and nothing else may stay.
"""
import pytest
import torch

import fine_grained_mixture_gb300 as moe
from fine_grained_mixture_gb300 import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

MIB = 1 << 20


@pytest.mark.parametrize("mode", ["tc", "tr"])
def test_forward_leaves_only_H_and_routing_metadata(mode):
    w = synth.WORKLOADS["fine7b"]
    g = to_dev(synth.make_inputs(w, 5))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    before = torch.cuda.memory_allocated()
    rt = moe.moe_route(g["logits"], w.K, mode)
    O, H = moe.moe_forward(g["X"], g["W1"], g["W2"], rt)
    del O
    torch.cuda.synchronize()
    grown = torch.cuda.memory_allocated() - before

    kept = [H, rt.topk_idx, rt.topk_score, rt.tc_counts, rt.counts, rt.offsets, rt.tile_offsets, rt.row_token,
            rt.row_slot, rt.row_score, rt.status, rt.ws]
    expected = sum(t.numel() * t.element_size() for t in kept)
    # the allocator rounds each block up (512 bytes; a split of a larger segment may keep up to 1 MiB more)
    assert expected <= grown <= expected + len(kept) * MIB, (grown, expected)

    code, P = rt.device_status()
    assert code == 0
    if mode == "tc":
        assert H.numel() * 2 == 4 * w.T * w.K * w.n  # the 4TKn term: P_cap = TK rows of 2n bf16
    else:
        assert P * 2 * w.n * 2 <= H.numel() * 2      # H is sized for the capacity; P rows are live
    transient = moe.moe_forward_workspace_size(w.T, w.d, w.n, w.E, w.K, rt.p_cap)
    assert transient > 64 * MIB                      # a leak of the workspace would exceed the slack above
