"""The Python binding's argument marshalling, on the CPU.

Shape-only ("meta") tensors stand in for device tensors, and a recording stand-in for the library's compute entry
points replaces the launches (the size and capacity queries still go to libmoe.so).  Checked here: valid calls
reach the library with the sizes the C ABI expects, and calls whose buffers would let the library read or write
out of bounds (a short buffer, a transposed weight, routing buffers made for another shape or mode, tensors on
different devices) raise before anything is launched.
"""
import contextlib

import pytest
import torch

import fine_grained_mixture_gb300 as moe
from fine_grained_mixture_gb300 import moe as binding

COMPUTE = ("moe_route_ex", "moe_forward_ex", "moe_backward_ex", "moe_router_forward", "moe_router_backward",
           "moe_get_status")
T, d, n, E, K = 300, 512, 128, 8, 2  # d != 2n, so a transposed W1 has another shape
bf, f32 = torch.bfloat16, torch.float32


class _Recorder:
    def __init__(self, real):
        self.real, self.calls = real, []

    def __getattr__(self, name):
        if name in COMPUTE:
            return lambda *args: (self.calls.append((name, args)), 0)[1]
        return getattr(self.real, name)


@pytest.fixture
def lib(monkeypatch):
    rec = _Recorder(binding.library())
    monkeypatch.setattr(binding, "_LIB", rec)
    monkeypatch.setattr(binding, "_stream", lambda stream=None, device=None: None)
    monkeypatch.setattr(torch.cuda, "device", lambda dev: contextlib.nullcontext())
    real_device = binding._device

    def meta_device(**tensors):
        try:
            return real_device(**tensors)
        except ValueError as e:
            if "expected CUDA" in str(e):
                return torch.device("meta")
            raise
    monkeypatch.setattr(binding, "_device", meta_device)
    return rec


def meta(*shape, dtype=bf):
    return torch.empty(shape, dtype=dtype, device="meta")


def layer(mode="tc"):
    rt = moe.Routing(T, E, K, mode, "meta")
    return rt, meta(T, d), meta(E, d, 2 * n), meta(E, n, d)


def ints(args, first, count):
    return tuple(int(a) for a in args[first:first + count])


def test_valid_calls_reach_the_library_with_the_abi_sizes(lib):
    rt, X, W1, W2 = layer("tr")
    moe.moe_route(meta(T, E, dtype=f32), K, "tr", routing=rt)
    O, H = moe.moe_forward(X, W1, W2, rt)
    moe.moe_backward(meta(T, d), X, W1, W2, H, rt)
    Wr = meta(d, E)
    z = moe.moe_router_forward(X, Wr)
    moe.moe_router_backward(meta(rt.p_cap, dtype=f32), rt, z, X, Wr, meta(T, d))
    names = [c[0] for c in lib.calls]
    assert names == ["moe_route_ex", "moe_forward_ex", "moe_backward_ex", "moe_router_forward", "moe_router_backward"]
    args = dict(lib.calls)
    assert ints(args["moe_route_ex"], 2, 4) == (T, E, K, moe.MOE_ROUTE_TR)
    assert ints(args["moe_forward_ex"], 4, 6) == (T, d, n, E, K, rt.p_cap)
    assert ints(args["moe_backward_ex"], 6, 6) == (T, d, n, E, K, rt.p_cap)
    assert ints(args["moe_router_forward"], 2, 3) == (T, d, E)
    assert ints(args["moe_router_backward"], 5, 6) == (T, d, E, K, moe.MOE_ROUTE_TR, rt.p_cap)
    assert tuple(O.shape) == (T, d) and tuple(H.shape) == (rt.p_cap, 2 * n) and tuple(z.shape) == (T, E)


def test_routing_buffers_must_match_the_call(lib):
    rt = moe.Routing(T, E, K, "tc", "meta")
    z = meta(T, E, dtype=f32)
    with pytest.raises(ValueError, match="routing buffers"):
        moe.moe_route(z, K, "tr", routing=rt)          # token rounding needs the larger row capacity
    with pytest.raises(ValueError, match="routing buffers"):
        moe.moe_route(z, K + 1, "tc", routing=rt)
    with pytest.raises(ValueError, match="routing buffers"):
        moe.moe_route(meta(T + 1, E, dtype=f32), K, "tc", routing=rt)
    _, X, W1, W2 = layer()
    with pytest.raises(ValueError, match="routing buffers"):
        moe.moe_forward(meta(T - 1, d), W1, W2, rt)
    with pytest.raises(ValueError, match="unknown routing mode"):
        moe.moe_route(z, K, "topk")
    assert lib.calls == []


def test_weight_shapes_are_checked(lib):
    rt, X, W1, W2 = layer()
    with pytest.raises(ValueError, match="W2"):
        moe.moe_forward(X, W1, meta(E, d, n), rt)                  # W2 transposed
    with pytest.raises(ValueError, match="W1"):
        moe.moe_forward(X, meta(E, 2 * n, d), W2, rt)               # W1 transposed
    with pytest.raises(ValueError, match="Wr"):
        moe.moe_router_forward(X, meta(E, d))                       # W_r transposed
    with pytest.raises(ValueError, match="dimensions"):
        moe.moe_forward(X.reshape(-1), W1, W2, rt)
    assert lib.calls == []


@pytest.mark.parametrize("name,shape,dtype", [
    ("O", (T - 1, d), bf), ("H", (10, 2 * n), bf), ("ws", (16,), torch.uint8), ("ws", (1 << 24,), f32),
])
def test_short_or_mistyped_forward_buffers_are_rejected(lib, name, shape, dtype):
    rt, X, W1, W2 = layer()
    with pytest.raises(ValueError, match=name):
        moe.moe_forward(X, W1, W2, rt, **{name: meta(*shape, dtype=dtype)})
    assert lib.calls == []


@pytest.mark.parametrize("name,shape,dtype", [
    ("dX", (T, d - 1), bf), ("dW1", (E - 1, d, 2 * n), bf), ("dW2", (E, n, d - 1), bf), ("dS", (T * K,), bf),
    ("ws", (64,), torch.uint8),
])
def test_short_or_mistyped_backward_buffers_are_rejected(lib, name, shape, dtype):
    rt, X, W1, W2 = layer("tr")
    H = meta(rt.p_cap, 2 * n)
    with pytest.raises(ValueError, match=name):
        moe.moe_backward(meta(T, d), X, W1, W2, H, rt, **{name: meta(*shape, dtype=dtype)})
    with pytest.raises(ValueError, match="H"):
        moe.moe_backward(meta(T, d), X, W1, W2, meta(T * K, 2 * n), rt)   # H sized for token choice, not rounding
    assert lib.calls == []


def test_router_backward_buffers_are_checked(lib):
    rt, X, _, _ = layer("tr")
    Wr, z, dX = meta(d, E), meta(T, E, dtype=f32), meta(T, d)
    with pytest.raises(ValueError, match="dS"):
        moe.moe_router_backward(meta(T * K, dtype=f32), rt, z, X, Wr, dX)   # rows of token choice only
    with pytest.raises(ValueError, match="dlogits"):
        moe.moe_router_backward(meta(rt.p_cap, dtype=f32), rt, z, X, Wr, dX, dlogits=meta(T, E - 1, dtype=f32))
    with pytest.raises(ValueError, match="routing buffers"):
        moe.moe_router_backward(meta(rt.p_cap, dtype=f32), rt, z, X, meta(d, 2 * E), dX)
    assert lib.calls == []


def test_tensors_on_different_devices_are_rejected():
    with pytest.raises(ValueError, match="different devices"):
        binding._device(X=torch.empty(4), W=torch.empty(4, device="meta"))
    with pytest.raises(ValueError, match="expected CUDA"):
        binding._device(X=torch.empty(4), W=None)
