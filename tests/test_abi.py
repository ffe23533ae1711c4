"""The C ABI without a GPU: the library loads, exports every function include/moe.h declares, and its
host-side validation returns the documented status codes (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import fine_grained_mixture_gb300 as moe
from fine_grained_mixture_gb300 import build as b

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    b.build()
    return moe.library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for f in ("moe_route", "moe_forward", "moe_backward", "moe_route_capacity", "moe_get_status"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    missing = [f for f in declared_functions() if not hasattr(lib, f)]
    assert not missing, missing


def declared_prototypes():
    """{name: (return type, [parameter declarations])} of every function include/moe.h declares."""
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for ret, name, params in re.findall(r"^\s*((?:const\s+)?[A-Za-z_][\w\s\*]*?)\b(moe_\w+)\s*\(([^)]*)\)\s*;",
                                        text, flags=re.M):
        plist = [p.strip() for p in params.split(",") if p.strip() and p.strip() != "void"]
        out[name] = (" ".join(ret.split()), plist)
    return out


_C_TO_CTYPES = {"int": ctypes.c_int, "unsigned": ctypes.c_uint, "size_t": ctypes.c_size_t,
                "int32_t": ctypes.c_int32, "uint64_t": ctypes.c_uint64, "double": ctypes.c_double}


def test_binding_signatures_match_the_header(lib):
    """Every function the binding declares to ctypes takes the header's number of arguments, passes pointers
    where the header has pointers and the header's scalar type elsewhere, and returns the header's type."""
    protos = declared_prototypes()
    checked = 0
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        checked += 1
        assert len(fn.argtypes) == len(params), (name, params, fn.argtypes)
        for decl, ct in zip(params, fn.argtypes):
            if "*" in decl:
                assert ct is ctypes.c_void_p or ct is ctypes.c_char_p or hasattr(ct, "_type_") and \
                    issubclass(ct, ctypes._Pointer), (name, decl, ct)
            else:
                base = decl.replace("const", "").split()[0]
                assert ct is _C_TO_CTYPES[base], (name, decl, ct)
        want = {"int": ctypes.c_int, "uint64_t": ctypes.c_uint64, "const char *": ctypes.c_char_p}[ret]
        assert fn.restype is want, (name, ret, fn.restype)
    assert checked >= 20, checked


def test_capacity_and_workspace_queries(lib):
    assert moe.moe_route_capacity(24576, 128, 8, "tc") == 24576 * 8
    assert moe.moe_route_capacity(24576, 128, 8, "tr") == 24576 * 8 + 128 * 64
    for mode in ("tr_up", "tr_stoch"):
        assert moe.moe_route_capacity(24576, 128, 8, mode) == 24576 * 8 + 128 * 127
    for mode in ("tr_down", "ec"):
        assert moe.moe_route_capacity(24576, 128, 8, mode) == 24576 * 8
    tc_ws = moe.moe_route_workspace_size(4096, 64, 8, "tc")
    for mode in ("tr", "tr_up", "tr_down", "tr_stoch", "ec"):
        assert moe.moe_route_workspace_size(4096, 64, 8, mode) >= tc_ws + 4096 * 64 * 4   # + expert-major keys
    p = moe.moe_route_capacity(512, 8, 2, "tc")
    fw = moe.moe_forward_workspace_size(512, 256, 128, 8, 2, p)
    assert fw >= p * 128 * 2 + 512 * 256 * 4
    bw = moe.moe_backward_workspace_size(512, 256, 128, 8, 2, p)
    assert bw >= p * 256 * 2 + p * 128 * 2 + 512 * 256 * 4


@pytest.mark.parametrize("args,code", [
    ((0, 8, 2, 0), 1), ((16, 8, 9, 0), 1), ((16, 8, 2, 7), 1), ((16, 8, 2, 6), 1), ((16, 8, 2, -1), 1),
    ((16, 2000, 2, 0), 2), ((16, 64, 40, 0), 2), ((60000, 8, 2, 1), 2), ((60000, 8, 2, 5), 2),
    # the selection modes hold one expert's keys for every token on chip: T = 49152 is their largest count
    ((49152, 1024, 32, 1), 0), ((49153, 8, 2, 1), 2), ((49153, 8, 2, 4), 2), ((49153, 1024, 32, 0), 0),
])
def test_route_validation(lib, args, code):
    out = ctypes.c_size_t(0)
    assert lib.moe_route_capacity(*args, ctypes.byref(out)) == code


@pytest.mark.parametrize("shape,code", [
    ((512, 200, 128, 8, 2, 1024), 2),     # d not a multiple of 256
    ((512, 256, 100, 8, 2, 1024), 2),     # n not a multiple of 128
    ((512, 256, 128, 8, 2, 1000), 1),     # capacity below T*K
    ((512, 256, 128, 8, 9, 4096), 1),     # K > E
])
def test_layer_validation(lib, shape, code):
    out = ctypes.c_size_t(0)
    assert lib.moe_forward_workspace_size(*shape, ctypes.byref(out)) == code
    assert lib.moe_backward_workspace_size(*shape, ctypes.byref(out)) == code


def test_deterministic_flag_queries(lib):
    p = moe.moe_route_capacity(512, 8, 2, "tc")
    base_f = moe.moe_forward_workspace_size(512, 256, 128, 8, 2, p)
    base_b = moe.moe_backward_workspace_size(512, 256, 512, 8, 2, p)
    assert moe.moe_forward_workspace_size(512, 256, 128, 8, 2, p, moe.MOE_FLAG_DETERMINISTIC) >= base_f + 512 * 256 * 4
    # 64-bit dX accumulator and the dS partials of two 256-wide column tiles
    assert moe.moe_backward_workspace_size(512, 256, 512, 8, 2, p, moe.MOE_FLAG_DETERMINISTIC) >= \
        base_b + 512 * 256 * 4 + p * 2 * 4
    out = ctypes.c_size_t(0)
    assert lib.moe_forward_workspace_size_ex(512, 256, 128, 8, 2, p, 4, ctypes.byref(out)) == 1   # unknown flag
    assert lib.moe_backward_workspace_size_ex(512, 256, 128, 8, 2, p, 6, ctypes.byref(out)) == 1
    # A kept on chip: the forward workspace holds no A [P_cap, n] bf16; the backward does not take the flag
    assert moe.moe_forward_workspace_size(512, 256, 128, 8, 2, p, moe.MOE_FLAG_A_FROM_H) == base_f - p * 128 * 2
    assert lib.moe_backward_workspace_size_ex(512, 256, 128, 8, 2, p, moe.MOE_FLAG_A_FROM_H, ctypes.byref(out)) == 1
    assert lib.moe_strerror(9) == b"value beyond the deterministic accumulator's range"


def test_null_arguments_rejected_before_any_device_work(lib):
    r = moe.moe.moe_routing()
    assert lib.moe_route(None, 16, 8, 2, 0, ctypes.byref(r), None, 0, None, None) == 1
    # stochastic rounding without its uniforms: rejected on the host (the pointers are never dereferenced)
    dummy = moe.moe.moe_routing(*([16] * 10))
    assert lib.moe_route_ex(ctypes.c_void_p(16), None, 16, 8, 2, 4, ctypes.byref(dummy), None, 0, None, None) == 1
    assert lib.moe_route(ctypes.c_void_p(16), 16, 8, 2, 4, ctypes.byref(dummy), None, 0, None, None) == 1
    assert lib.moe_forward(None, None, None, ctypes.byref(r), 512, 256, 128, 8, 2, 1024, None, None, None, 0,
                           None) == 1
    assert lib.moe_strerror(6) == b"device pipeline wait timed out"


def test_router_validation(lib):
    out = ctypes.c_size_t(0)
    assert lib.moe_router_backward_workspace_size(24576, 1536, 128, ctypes.byref(out)) == 0
    # bf16 dz [T, E] plus up to 32 fp32 partials of dW_r [d, E]
    assert out.value >= 24576 * 128 * 2 + 32 * 1536 * 128 * 4
    assert lib.moe_router_backward_workspace_size(64, 256, 12, ctypes.byref(out)) == 2   # E % 8 != 0
    assert lib.moe_router_backward_workspace_size(64, 200, 16, ctypes.byref(out)) == 2   # d % 256 != 0
    assert lib.moe_router_backward_workspace_size(0, 256, 16, ctypes.byref(out)) == 1
    assert lib.moe_router_backward_workspace_size(64, 256, 16, None) == 1
    # null tensors are rejected before any device work
    assert lib.moe_router_forward(None, None, 64, 256, 16, None, None, None) == 1
    assert lib.moe_router_forward(ctypes.c_void_p(16), ctypes.c_void_p(16), 64, 256, 12, ctypes.c_void_p(16), None,
                                  None) == 2
    r = moe.moe.moe_routing()
    assert lib.moe_router_backward(None, ctypes.byref(r), None, None, None, 64, 256, 16, 2, 0, 128, None, None, None,
                                   None, 0, None) == 1


def test_deterministic_entry_points_reject_unknown_flags(lib):
    dummy = moe.moe.moe_routing(*([16] * 10))
    p = ctypes.c_void_p(16)
    assert lib.moe_forward_ex(p, p, p, ctypes.byref(dummy), 512, 256, 128, 8, 2, 1024, p, p, p, 1 << 30, 4,
                              None) == 1
    assert lib.moe_backward_ex(p, p, p, p, p, ctypes.byref(dummy), 512, 256, 128, 8, 2, 1024, p, p, p, p, p, 1 << 30,
                               8, None) == 1
