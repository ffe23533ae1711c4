"""GB300-native (sm_103a) fine-grained MoE expert layer: routing, forward and backward behind a C ABI.

The compute runs in libmoe.so (hand-written CUDA); ``moe`` is the thin ctypes binding over it.
"""
from .moe import (M_TILE, MODES, MOE_FLAG_A_FROM_H, MOE_FLAG_DETERMINISTIC, MOE_ROUTE_EC, MOE_ROUTE_TC, MOE_ROUTE_TR, MOE_ROUTE_TR_DOWN,
                  MOE_ROUTE_TR_STOCHASTIC, MOE_ROUTE_TR_UP, MoeError, Routing, kernel_launch_count, library,
                  moe_backward, moe_backward_workspace_size, moe_forward, moe_forward_workspace_size, moe_route,
                  moe_route_capacity, moe_route_workspace_size, moe_router_backward, moe_router_forward,
                  profile_enable, profile_summary, selftest_bounded_wait)

__all__ = ["M_TILE", "MODES", "MOE_FLAG_A_FROM_H", "MOE_FLAG_DETERMINISTIC", "MOE_ROUTE_EC", "MOE_ROUTE_TC", "MOE_ROUTE_TR", "MOE_ROUTE_TR_DOWN",
           "MOE_ROUTE_TR_STOCHASTIC", "MOE_ROUTE_TR_UP", "MoeError", "Routing", "kernel_launch_count", "library",
           "moe_backward", "moe_backward_workspace_size", "moe_forward", "moe_forward_workspace_size", "moe_route",
           "moe_route_capacity", "moe_route_workspace_size", "moe_router_backward", "moe_router_forward",
           "profile_enable", "profile_summary", "selftest_bounded_wait"]

from . import dp  # noqa: E402  (data parallelism: token shards and the weight-gradient all-reduce)
