"""GB300-native MoE token routing: gate -> dispatch layout -> dispatch ->
combine, as hand-written sm_103a CUDA kernels behind a C ABI
(include/moe_route.h, libmoeroute.so), with a thin ctypes binding.

PyTorch supplies device memory and streams only.  The routing work runs in
the library's kernels; importing the binding fails loudly if the library has
not been built (``build()``).
"""
from . import _build
from .abi import (MOE_ERR_CUDA, MOE_ERR_DEVICE_DATA, MOE_ERR_INVALID_ARG, MOE_ERR_TIMEOUT,
                  MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE_TOO_SMALL, MOE_FP8_GLOBAL, MOE_FP8_PER_EXPERT,
                  MOE_FP8_PER_TOKEN, MOE_OK, MOE_SOFTMAX_TOPK, MOE_TOPK_SOFTMAX, Layout, MoeError,
                  alloc_workspace, moe_combine, moe_combine_backward, moe_combine_fp8, moe_dispatch,
                  moe_dispatch_backward, moe_dispatch_layout, moe_gate, moe_gate_backward, moe_get_status,
                  moe_quantize_rows, moe_route, moe_rows_max, moe_workspace_init, moe_workspace_size)
from .pipeline import RouteGraph, RoutePipeline, RoutePlan, RouteShape


def build(force: bool = False) -> str:
    """Compile libmoeroute.so for sm_103a (in-tree)."""
    return _build.build(force=force)


__all__ = [
    "build", "RoutePlan", "RoutePipeline", "RouteGraph", "RouteShape", "Layout", "MoeError", "alloc_workspace",
    "moe_gate", "moe_dispatch_layout", "moe_dispatch", "moe_combine", "moe_get_status", "moe_route",
    "moe_quantize_rows", "moe_combine_fp8", "moe_combine_backward", "moe_dispatch_backward",
    "moe_gate_backward", "MOE_FP8_PER_TOKEN", "MOE_FP8_PER_EXPERT", "MOE_FP8_GLOBAL",
    "moe_workspace_size", "moe_workspace_init", "moe_rows_max",
    "MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE_TOO_SMALL",
    "MOE_ERR_CUDA", "MOE_ERR_TIMEOUT", "MOE_ERR_DEVICE_DATA", "MOE_TOPK_SOFTMAX", "MOE_SOFTMAX_TOPK",
]
