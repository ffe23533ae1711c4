"""Thin Python binding of libmoe (the C ABI in include/moe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module allocates the caller-owned
device buffers with torch, passes raw pointers and the current CUDA stream, and turns status codes into
exceptions.  There is no fallback: if libmoe.so is missing or the device is not a GB300 the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MOE_ROUTE_TC = 0
MOE_ROUTE_TR = 1
MOE_ROUTE_TR_UP = 2
MOE_ROUTE_TR_DOWN = 3
MOE_ROUTE_TR_STOCHASTIC = 4
MOE_ROUTE_EC = 5
M_TILE = 128
STATUS_WORDS = 4
MOE_FLAG_DETERMINISTIC = 1  # bitwise-reproducible aggregation (fixed-point accumulators)
MOE_FLAG_A_FROM_H = 2  # the down-projection recomputes A = SwiGLU(H) on chip; A is never written
# token choice; token rounding to the nearest tile, always up, always down, stochastically; expert choice
MODES = {"tc": MOE_ROUTE_TC, "tr": MOE_ROUTE_TR, "tr_up": MOE_ROUTE_TR_UP, "tr_down": MOE_ROUTE_TR_DOWN,
         "tr_stoch": MOE_ROUTE_TR_STOCHASTIC, "ec": MOE_ROUTE_EC}

ERRORS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_WORKSPACE",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_NONFINITE_LOGITS", 6: "MOE_ERR_DEVICE_TIMEOUT", 7: "MOE_ERR_BAD_METADATA",
    8: "MOE_ERR_DEVICE", 9: "MOE_ERR_RANGE",
}


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {ERRORS.get(code, code)}"
        if code == 4 and _LIB is not None:
            msg += f" (cuda error {_LIB.moe_last_cuda_error()})"
        super().__init__(msg)


class moe_routing(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "topk_idx", "topk_score", "tc_counts", "counts", "offsets", "tile_offsets",
        "row_token", "row_slot", "row_score", "status")]


_LIB = None
_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p


def library() -> ctypes.CDLL:
    """Load libmoe.so from the package directory (built by __graft_entry__.build())."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libmoe.so is not built ({_build.LIB}); run __graft_entry__.build()")
    lib = ctypes.CDLL(_build.LIB)
    sz = ctypes.POINTER(_c_size)
    lib.moe_route_capacity.argtypes = [_c_int, _c_int, _c_int, _c_int, sz]
    lib.moe_route_workspace_size.argtypes = [_c_int, _c_int, _c_int, _c_int, sz]
    lib.moe_route.argtypes = [_vp, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(moe_routing), _vp, _c_size,
                              ctypes.POINTER(ctypes.c_int32), _vp]
    lib.moe_route_ex.argtypes = [_vp, _vp, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(moe_routing), _vp, _c_size,
                                 ctypes.POINTER(ctypes.c_int32), _vp]
    lib.moe_forward_workspace_size.argtypes = [_c_int] * 5 + [_c_size, sz]
    lib.moe_forward_workspace_size_ex.argtypes = [_c_int] * 5 + [_c_size, ctypes.c_uint, sz]
    lib.moe_backward_workspace_size_ex.argtypes = [_c_int] * 5 + [_c_size, ctypes.c_uint, sz]
    lib.moe_forward_ex.argtypes = [_vp, _vp, _vp, ctypes.POINTER(moe_routing)] + [_c_int] * 5 + [
        _c_size, _vp, _vp, _vp, _c_size, ctypes.c_uint, _vp]
    lib.moe_backward_ex.argtypes = [_vp] * 5 + [ctypes.POINTER(moe_routing)] + [_c_int] * 5 + [_c_size] + [_vp] * 5 + [
        _c_size, ctypes.c_uint, _vp]
    lib.moe_forward.argtypes = [_vp, _vp, _vp, ctypes.POINTER(moe_routing)] + [_c_int] * 5 + [_c_size, _vp, _vp, _vp,
                                                                                              _c_size, _vp]
    lib.moe_backward_workspace_size.argtypes = [_c_int] * 5 + [_c_size, sz]
    lib.moe_backward.argtypes = [_vp] * 5 + [ctypes.POINTER(moe_routing)] + [_c_int] * 5 + [_c_size] + [_vp] * 5 + [
        _c_size, _vp]
    lib.moe_router_forward.argtypes = [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp]
    lib.moe_router_backward_workspace_size.argtypes = [_c_int, _c_int, _c_int, sz]
    lib.moe_router_backward.argtypes = [_vp, ctypes.POINTER(moe_routing), _vp, _vp, _vp] + [_c_int] * 5 + [
        _c_size, _vp, _vp, _vp, _vp, _c_size, _vp]
    lib.moe_get_status.argtypes = [ctypes.POINTER(moe_routing), ctypes.POINTER(ctypes.c_int32),
                                   ctypes.POINTER(ctypes.c_int32), _vp]
    lib.moe_strerror.argtypes = [_c_int]
    lib.moe_strerror.restype = ctypes.c_char_p
    lib.moe_last_cuda_error.argtypes = []
    lib.moe_kernel_launch_count.argtypes = []
    lib.moe_kernel_launch_count.restype = ctypes.c_uint64
    lib.moe_selftest_bounded_wait.argtypes = [_vp, _vp]
    lib.moe_selftest_bounded_wait.restype = _c_int
    lib.moe_profile_enable.argtypes = [_c_int]
    lib.moe_profile_count.argtypes = []
    lib.moe_profile_entry.argtypes = [_c_int, ctypes.c_char_p, _c_size, ctypes.POINTER(_c_int),
                                      ctypes.POINTER(ctypes.c_double)]
    for f in ("moe_profile_enable", "moe_profile_count", "moe_profile_entry"):
        getattr(lib, f).restype = _c_int
    for f in ("moe_route_capacity", "moe_route_workspace_size", "moe_route", "moe_route_ex", "moe_forward_workspace_size",
              "moe_forward", "moe_backward_workspace_size", "moe_backward", "moe_get_status", "moe_last_cuda_error",
              "moe_router_forward", "moe_router_backward_workspace_size", "moe_router_backward",
              "moe_forward_workspace_size_ex", "moe_backward_workspace_size_ex", "moe_forward_ex", "moe_backward_ex"):
        getattr(lib, f).restype = _c_int
    _LIB = lib
    return lib


def selftest_bounded_wait(stream=None) -> int:
    """Run the bounded-wait self-test; returns the device status code it wrote (MOE_ERR_DEVICE_TIMEOUT = 6)."""
    lib = library()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(lib.moe_selftest_bounded_wait(_ptr(st), _stream(stream)), "moe_selftest_bounded_wait")
    torch.cuda.synchronize()
    return int(st.item())


def _check(code: int, where: str):
    if code != 0:
        raise MoeError(code, where)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None, device: torch.device | None = None):
    """The cudaStream_t of `stream`, else of the current stream of `device` (the current device by default)."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    if device is not None and s.device != device:
        raise ValueError(f"stream is on {s.device}, the tensors on {device}")
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, numel: int | None = None):
    """A contiguous tensor of `dtype` with at least `numel` elements (the library reads and writes that many)."""
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous {dtype} tensor, got {t.dtype} {tuple(t.shape)}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: needs {numel} elements, has {t.numel()}")


def _dims(t: torch.Tensor, name: str, ndim: int):
    if t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dimensions, got shape {tuple(t.shape)}")
    return tuple(t.shape)


def _device(**tensors) -> torch.device:
    """The one CUDA device that every given tensor (None entries skipped) lives on; calls run with it current."""
    devs: dict = {}
    for name, t in tensors.items():
        if t is not None:
            devs.setdefault(t.device, name)
    if len(devs) != 1:
        raise ValueError("tensors on different devices: " + ", ".join(f"{n} on {d}" for d, n in devs.items()))
    dev = next(iter(devs))
    if dev.type != "cuda":
        raise ValueError(f"expected CUDA tensors, got tensors on {dev}")
    return dev


def _mode(mode) -> int:
    if isinstance(mode, str):
        if mode not in MODES:
            raise ValueError(f"unknown routing mode {mode!r}; one of {sorted(MODES)}")
        return MODES[mode]
    return int(mode)


def _same_routing(routing: "Routing", T: int, E: int):
    if (routing.T, routing.E) != (T, E):
        raise ValueError(f"routing buffers were made for T={routing.T}, E={routing.E}; the tensors have T={T}, E={E}")


def moe_route_capacity(T: int, E: int, K: int, mode="tc") -> int:
    out = _c_size(0)
    _check(library().moe_route_capacity(T, E, K, _mode(mode), ctypes.byref(out)), "moe_route_capacity")
    return out.value


def moe_route_workspace_size(T: int, E: int, K: int, mode="tc") -> int:
    out = _c_size(0)
    _check(library().moe_route_workspace_size(T, E, K, _mode(mode), ctypes.byref(out)), "moe_route_workspace_size")
    return out.value


def moe_forward_workspace_size(T, d, n, E, K, p_cap, flags: int = 0) -> int:
    out = _c_size(0)
    _check(library().moe_forward_workspace_size_ex(T, d, n, E, K, p_cap, flags, ctypes.byref(out)),
           "moe_forward_workspace_size_ex")
    return out.value


def moe_backward_workspace_size(T, d, n, E, K, p_cap, flags: int = 0) -> int:
    out = _c_size(0)
    _check(library().moe_backward_workspace_size_ex(T, d, n, E, K, p_cap, flags, ctypes.byref(out)),
           "moe_backward_workspace_size_ex")
    return out.value


class Routing:
    """Caller-owned routing metadata buffers (torch tensors on one device) and the C struct over them."""

    def __init__(self, T: int, E: int, K: int, mode="tc", device="cuda"):
        self.T, self.E, self.K, self.mode = T, E, K, _mode(mode)
        self.p_cap = moe_route_capacity(T, E, K, self.mode)
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.topk_idx = torch.empty(T * K, **i32)
        self.topk_score = torch.empty(T * K, **f32)
        self.tc_counts = torch.empty(E, **i32)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.tile_offsets = torch.empty(E + 1, **i32)
        self.row_token = torch.empty(self.p_cap, **i32)
        self.row_slot = torch.empty(self.p_cap, **i32)
        self.row_score = torch.empty(self.p_cap, **f32)
        self.status = torch.zeros(STATUS_WORDS, **i32)
        self.ws = torch.empty(moe_route_workspace_size(T, E, K, self.mode), dtype=torch.uint8, device=device)
        self.struct = moe_routing(*[t.data_ptr() for t in (
            self.topk_idx, self.topk_score, self.tc_counts, self.counts, self.offsets, self.tile_offsets,
            self.row_token, self.row_slot, self.row_score, self.status)])

    def device_status(self, stream=None):
        """(device error code, P) after synchronising the stream."""
        code, P = ctypes.c_int32(0), ctypes.c_int32(0)
        dev = _device(status=self.status)
        with torch.cuda.device(dev):
            _check(library().moe_get_status(ctypes.byref(self.struct), ctypes.byref(code), ctypes.byref(P),
                                            _stream(stream, dev)), "moe_get_status")
        return code.value, P.value


def moe_route(logits: torch.Tensor, K: int, mode="tc", routing: Routing | None = None, want_P=False, stream=None,
              uniforms: torch.Tensor | None = None):
    """Routing metadata for fp32 logits [T, E]; returns the Routing (and P when want_P).

    uniforms: fp32 [E] draws in [0, 1) for stochastic rounding ("tr_stoch"); other modes ignore them.
    routing: buffers from an earlier call (or Routing(...)) to fill again; they must match T, E, K and mode."""
    T, E = _dims(logits, "logits", 2)
    _need(logits, "logits", torch.float32)
    m = _mode(mode)
    if routing is None:
        routing = Routing(T, E, K, m, logits.device)
    elif (routing.T, routing.E, routing.K, routing.mode) != (T, E, K, m):
        raise ValueError(f"routing buffers were made for T={routing.T}, E={routing.E}, K={routing.K}, mode "
                         f"{routing.mode}; this call has T={T}, E={E}, K={K}, mode {m}")
    if uniforms is not None:
        _need(uniforms, "uniforms", torch.float32, E)
    dev = _device(logits=logits, routing=routing.status, uniforms=uniforms)
    P = ctypes.c_int32(0)
    with torch.cuda.device(dev):
        _check(library().moe_route_ex(_ptr(logits), _ptr(uniforms), T, E, K, routing.mode,
                                      ctypes.byref(routing.struct), _ptr(routing.ws), routing.ws.numel(),
                                      ctypes.byref(P) if want_P else None, _stream(stream, dev)), "moe_route_ex")
    return (routing, P.value) if want_P else routing


def _layer_dims(X, W1, W2, routing: Routing):
    """(T, d, E, n) from X [T, d], W1 [E, d, 2n], W2 [E, n, d], checked against each other and the routing."""
    T, d = _dims(X, "X", 2)
    E, d1, n2 = _dims(W1, "W1", 3)
    if d1 != d or n2 % 2:
        raise ValueError(f"W1: expected [E, {d}, 2n], got {(E, d1, n2)}")
    n = n2 // 2
    if _dims(W2, "W2", 3) != (E, n, d):
        raise ValueError(f"W2: expected {(E, n, d)}, got {tuple(W2.shape)}")
    _same_routing(routing, T, E)
    return T, d, E, n


def moe_forward(X, W1, W2, routing: Routing, O=None, H=None, ws=None, stream=None, deterministic=False,
                a_from_h=False):
    """O = sum_k s_k SwiGLU(X W1_e) W2_e; returns (O [T, d] bf16, H [P_cap, 2n] bf16).

    deterministic: fixed-point aggregation, bitwise identical results on every run.
    a_from_h: the down-projection recomputes A = SwiGLU(H) from the cached H on chip (A is never written)."""
    T, d, E, n = _layer_dims(X, W1, W2, routing)
    n2 = 2 * n
    K, p_cap = routing.K, routing.p_cap
    bf = torch.bfloat16
    _need(X, "X", bf)
    _need(W1, "W1", bf)
    _need(W2, "W2", bf)
    O = torch.empty((T, d), dtype=bf, device=X.device) if O is None else O
    H = torch.empty((p_cap, n2), dtype=bf, device=X.device) if H is None else H
    flags = (MOE_FLAG_DETERMINISTIC if deterministic else 0) | (MOE_FLAG_A_FROM_H if a_from_h else 0)
    need = moe_forward_workspace_size(T, d, n, E, K, p_cap, flags)
    ws = torch.empty(need, dtype=torch.uint8, device=X.device) if ws is None else ws
    _need(O, "O", bf, T * d)
    _need(H, "H", bf, p_cap * n2)
    _need(ws, "ws", torch.uint8, need)
    dev = _device(X=X, W1=W1, W2=W2, routing=routing.status, O=O, H=H, ws=ws)
    with torch.cuda.device(dev):
        _check(library().moe_forward_ex(_ptr(X), _ptr(W1), _ptr(W2), ctypes.byref(routing.struct), T, d, n, E, K,
                                        p_cap, _ptr(O), _ptr(H), _ptr(ws), ws.numel(), flags, _stream(stream, dev)),
               "moe_forward_ex")
    return O, H


def moe_backward(dO, X, W1, W2, H, routing: Routing, dX=None, dW1=None, dW2=None, dS=None, ws=None, stream=None,
                 deterministic=False):
    """Gradients for upstream dO; returns (dX [T, d], dW1 [E, d, 2n], dW2 [E, n, d], dS [P_cap] fp32).

    deterministic: fixed-point aggregation of dX and ordered dS sums, bitwise identical results on every run."""
    T, d, E, n = _layer_dims(X, W1, W2, routing)
    n2 = 2 * n
    K, p_cap = routing.K, routing.p_cap
    bf = torch.bfloat16
    for t, name, numel in ((dO, "dO", T * d), (X, "X", None), (W1, "W1", None), (W2, "W2", None),
                           (H, "H", p_cap * n2)):
        _need(t, name, bf, numel)
    dev = X.device
    dX = torch.empty((T, d), dtype=bf, device=dev) if dX is None else dX
    dW1 = torch.empty((E, d, n2), dtype=bf, device=dev) if dW1 is None else dW1
    dW2 = torch.empty((E, n, d), dtype=bf, device=dev) if dW2 is None else dW2
    dS = torch.empty(p_cap, dtype=torch.float32, device=dev) if dS is None else dS
    flags = MOE_FLAG_DETERMINISTIC if deterministic else 0
    need = moe_backward_workspace_size(T, d, n, E, K, p_cap, flags)
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if ws is None else ws
    for t, name, dt, numel in ((dX, "dX", bf, T * d), (dW1, "dW1", bf, E * d * n2), (dW2, "dW2", bf, E * n * d),
                               (dS, "dS", torch.float32, p_cap), (ws, "ws", torch.uint8, need)):
        _need(t, name, dt, numel)
    dev = _device(dO=dO, X=X, W1=W1, W2=W2, H=H, routing=routing.status, dX=dX, dW1=dW1, dW2=dW2, dS=dS, ws=ws)
    with torch.cuda.device(dev):
        _check(library().moe_backward_ex(_ptr(dO), _ptr(X), _ptr(W1), _ptr(W2), _ptr(H),
                                         ctypes.byref(routing.struct), T, d, n, E, K, p_cap, _ptr(dX), _ptr(dW1),
                                         _ptr(dW2), _ptr(dS), _ptr(ws), ws.numel(), flags, _stream(stream, dev)),
               "moe_backward_ex")
    return dX, dW1, dW2, dS


def _router_dims(X, Wr):
    """(T, d, E) from X [T, d] and W_r [d, E]."""
    T, d = _dims(X, "X", 2)
    d1, E = _dims(Wr, "Wr", 2)
    if d1 != d:
        raise ValueError(f"Wr: expected [{d}, E], got {(d1, E)}")
    return T, d, E


def moe_router_forward(X, Wr, logits=None, status=None, stream=None):
    """Router logits = X W_r (X bf16 [T, d], W_r bf16 [d, E]); returns fp32 logits [T, E].

    status: optional int32 device tensor that receives MOE_ERR_DEVICE_TIMEOUT if a bounded wait runs out."""
    T, d, E = _router_dims(X, Wr)
    _need(X, "X", torch.bfloat16)
    _need(Wr, "Wr", torch.bfloat16)
    logits = torch.empty((T, E), dtype=torch.float32, device=X.device) if logits is None else logits
    _need(logits, "logits", torch.float32, T * E)
    if status is not None:
        _need(status, "status", torch.int32, 1)
    dev = _device(X=X, Wr=Wr, logits=logits, status=status)
    with torch.cuda.device(dev):
        _check(library().moe_router_forward(_ptr(X), _ptr(Wr), T, d, E, _ptr(logits), _ptr(status),
                                            _stream(stream, dev)), "moe_router_forward")
    return logits


def moe_router_backward(dS, routing: Routing, logits, X, Wr, dX, dlogits=None, dWr=None, ws=None, stream=None):
    """Router gradients through the gates (routing held fixed): returns (dlogits [T, E] fp32, dWr [d, E] fp32).

    dX (bf16 [T, d], the layer's input gradient from moe_backward) is updated in place with dz W_r^T."""
    T, d, E = _router_dims(X, Wr)
    _same_routing(routing, T, E)
    f32, bf = torch.float32, torch.bfloat16
    for t, name, dt, numel in ((dS, "dS", f32, routing.p_cap), (logits, "logits", f32, T * E), (X, "X", bf, None),
                               (Wr, "Wr", bf, None), (dX, "dX", bf, T * d)):
        _need(t, name, dt, numel)
    dev = X.device
    dlogits = torch.empty((T, E), dtype=f32, device=dev) if dlogits is None else dlogits
    dWr = torch.empty((d, E), dtype=f32, device=dev) if dWr is None else dWr
    out = _c_size(0)
    _check(library().moe_router_backward_workspace_size(T, d, E, ctypes.byref(out)), "moe_router_backward_workspace_size")
    ws = torch.empty(out.value, dtype=torch.uint8, device=dev) if ws is None else ws
    for t, name, dt, numel in ((dlogits, "dlogits", f32, T * E), (dWr, "dWr", f32, d * E),
                               (ws, "ws", torch.uint8, out.value)):
        _need(t, name, dt, numel)
    dev = _device(dS=dS, routing=routing.status, logits=logits, X=X, Wr=Wr, dX=dX, dlogits=dlogits, dWr=dWr, ws=ws)
    with torch.cuda.device(dev):
        _check(library().moe_router_backward(_ptr(dS), ctypes.byref(routing.struct), _ptr(logits), _ptr(X), _ptr(Wr),
                                             T, d, E, routing.K, routing.mode, routing.p_cap, _ptr(dlogits), _ptr(dX),
                                             _ptr(dWr), _ptr(ws), ws.numel(), _stream(stream, dev)),
               "moe_router_backward")
    return dlogits, dWr


def kernel_launch_count() -> int:
    return int(library().moe_kernel_launch_count())


def profile_enable(on: bool):
    """Start (clearing old results) or stop per-kernel CUDA-event timing inside the library."""
    _check(library().moe_profile_enable(1 if on else 0), "moe_profile_enable")


def profile_summary() -> dict:
    """{kernel name: (launches, total ms)} of the last finished profiling session."""
    lib = library()
    out = {}
    buf = ctypes.create_string_buffer(64)
    for i in range(lib.moe_profile_count()):
        n, ms = _c_int(0), ctypes.c_double(0.0)
        _check(lib.moe_profile_entry(i, buf, 64, ctypes.byref(n), ctypes.byref(ms)), "moe_profile_entry")
        out[buf.value.decode()] = (n.value, ms.value)
    return out
