"""moe_route_noalloc: routing for callers that may not allocate device memory (their host program's
allocator owns the device, or their path has a fixed memory budget).  It keeps its scratch in a static
array inside the library instead of a caller workspace; its results must equal moe_route's.

Collected last on purpose (file name), so a run that stops at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import fine_grained_mixture_gb300 as moe
from fine_grained_mixture_gb300.moe import moe_routing

pytestmark = pytest.mark.gpu

FIELDS = ("topk_idx", "tc_counts", "counts", "offsets", "tile_offsets", "row_token", "row_slot")


def _noalloc_fn():
    lib = moe.library()
    fn = lib.moe_route_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.POINTER(moe_routing), ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(fn, logits, K, mode):
    T, E = logits.shape
    out = moe.Routing(T, E, K, mode, logits.device)      # the caller still owns the outputs
    P = ctypes.c_int32(-1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(ctypes.c_void_p(logits.data_ptr()), T, E, K, out.mode, ctypes.byref(out.struct), ctypes.byref(P), stream)
    assert rc == 0, moe.moe.ERRORS.get(rc, rc)
    return out, P.value


def _same(a, b, P):
    for f in FIELDS:
        x, y = getattr(a, f), getattr(b, f)
        if f in ("row_token", "row_slot"):
            x, y = x[:P], y[:P]
        assert torch.equal(x, y), f
    np.testing.assert_allclose(a.topk_score.cpu().numpy(), b.topk_score.cpu().numpy(), rtol=1e-6, atol=0)
    np.testing.assert_allclose(a.row_score[:P].cpu().numpy(), b.row_score[:P].cpu().numpy(), rtol=1e-6, atol=0)


@pytest.mark.parametrize("mode", ["tc", "tr", "tr_up", "tr_down", "ec"])
@pytest.mark.parametrize("T,E,K", [(6144, 128, 8), (49152, 128, 8)])
def test_noalloc_matches_workspace_route_twice(mode, T, E, K):
    # at T=49152, E=128 the selection modes' full scratch (with the 25 MB expert-major key copy) exceeds the
    # static array, so the call takes the compact layout and reads the logits in place
    fn = _noalloc_fn()
    gen = torch.Generator().manual_seed(123)
    # two different inputs in a row: the second call must not see anything the first left behind
    for call in range(2):
        logits = torch.randn((T, E), generator=gen).cuda()
        if call == 1:
            logits[:, :4] += 3.0           # a different load pattern from the first call
        ref, P_ref = moe.moe_route(logits, K, mode, want_P=True)
        got, P = _call_noalloc(fn, logits, K, mode)
        torch.cuda.synchronize()
        assert P == P_ref
        code, _ = got.device_status()
        assert code == 0
        _same(got, ref, P)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fn = _noalloc_fn()
    T, E, K = 262144, 1024, 8               # needs more routing scratch than the static 16 MiB
    need = moe.moe_route_workspace_size(T, E, K, "tc")
    assert need > (16 << 20)
    dummy = torch.zeros(1, device="cuda")
    out = moe_routing()
    rc = fn(ctypes.c_void_p(dummy.data_ptr()), T, E, K, 0, ctypes.byref(out), None, None)
    assert rc == 3                            # MOE_ERR_WORKSPACE, before any device work


def test_noalloc_compact_layout_is_taken_by_every_selection_mode():
    # the shapes above exercise both scratch layouts: the full one fits at T=6144, only the compact one at 49152
    cap = 16 << 20
    for mode in ("tr", "tr_up", "tr_down", "ec"):
        assert moe.moe_route_workspace_size(6144, 128, 8, mode) <= cap
        assert moe.moe_route_workspace_size(49152, 128, 8, mode) > cap


def test_noalloc_rejects_stochastic_rounding():
    # stochastic rounding draws one uniform per expert, which only moe_route_ex takes
    fn = _noalloc_fn()
    logits = torch.randn((256, 16), device="cuda")
    out = moe.Routing(256, 16, 2, "tr", logits.device)
    rc = fn(ctypes.c_void_p(logits.data_ptr()), 256, 16, 2, moe.moe.MOE_ROUTE_TR_STOCHASTIC, ctypes.byref(out.struct),
            None, None)
    assert rc == 1                            # MOE_ERR_INVALID_ARG, before any device work
