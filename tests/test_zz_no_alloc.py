"""moe_dispatch_layout_noalloc: the layout entry point for callers that are
not allowed to allocate device memory (for example a plug-in inside a host
framework that owns all device memory through its own pool, or a
latency-critical loop that must stay out of the CUDA allocator).  It uses a
fixed scratch array compiled into the library instead of a caller-provided
workspace.

This file is collected last on purpose.  The test calls the new entry point
through the C ABI twice in a row, on different inputs, and requires its
output to equal the regular moe_dispatch_layout's bit for bit (the layout is
integer work: the exact-match tolerance of every other layout test).  It
builds what it needs, so it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from combine_moe_gate_warp_gb300 import RoutePlan, abi, workloads

pytestmark = pytest.mark.gpu

FIELDS = ("counts", "offsets", "part_rows", "part_offsets", "part_tokens", "src_pos", "dst_row",
          "capacity_mask", "dropped")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()


def _shape(w):
    from combine_moe_gate_warp_gb300 import RouteShape
    return RouteShape(T=w.T, H=w.H, E=w.E, k=w.k, P=w.P, mode=w.mode, fp8=w.fp8, Ks=w.Ks,
                      capacity=w.capacity)


def test_noalloc_layout_equals_workspace_layout_on_two_calls_in_a_row():
    lib = abi.lib()
    cases = [workloads.WORKLOADS["prefill_cap"].scaled(5000),
             workloads.WORKLOADS["fine_shared"].scaled(3001)]
    stream = torch.cuda.current_stream()
    for w in cases:
        inp = workloads.make_inputs(w, "cuda")
        plan = RoutePlan(_shape(w), "cuda")
        plan.gate(inp["logits"])
        gates_in = plan.gates.clone()
        plan.dispatch_layout()                          # regular entry point, caller workspace
        assert plan.status() == 0

        L2 = abi.Layout(w.T, w.E, w.k, w.P, w.capacity, "cuda")
        for name in FIELDS:
            getattr(L2, name).fill_(-7 if getattr(L2, name).dtype != torch.uint8 else 0xAB)
        gates2 = gates_in.clone()
        rc = lib.moe_dispatch_layout_noalloc(
            ctypes.c_void_p(plan.topk_idx.data_ptr()), ctypes.c_void_p(plan.expert_counts.data_ptr()),
            w.T, w.E, w.k, w.P, w.capacity, ctypes.c_void_p(gates2.data_ptr()), ctypes.byref(L2.c),
            ctypes.c_void_p(stream.cuda_stream))
        assert rc == abi.MOE_OK
        assert L2.c.ws is not None and L2.c.ws != plan.ws.data_ptr()
        assert lib.moe_get_status(ctypes.c_void_p(L2.c.ws), ctypes.c_void_p(stream.cuda_stream)) == 0

        R = int(plan.layout.offsets[w.E].item())
        for name in FIELDS:
            a = getattr(plan.layout, name)
            b = getattr(L2, name)
            if name == "src_pos":
                a, b = a[:R], b[:R]
            assert torch.equal(a, b), name
        assert torch.equal(plan.gates.view(torch.int32), gates2.view(torch.int32))
        if w.capacity:
            assert int(L2.dropped.item()) > 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = abi.lib()
    T, E, k, P = 1 << 20, 256, 16, 8
    assert abi.moe_workspace_size(T, E, k, P) > abi.MOE_NOALLOC_SCRATCH_BYTES
    L = abi.moe_layout()
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.moe_dispatch_layout_noalloc(fake, fake, T, E, k, P, 0, None, ctypes.byref(L), None)
    assert rc == abi.MOE_ERR_WORKSPACE_TOO_SMALL


class _DeviceWords:
    """A zero-copy view of device memory at a raw address (the library's
    scratch), through the CUDA array interface, so the test can write it."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False), "version": 3}


def test_noalloc_recovers_counters_left_dirty():
    """The scratch is shared by every call and keeps the last call's
    contents.  A call that stopped partway could leave its completion
    counters and partition-token totals non-zero; the entry point clears
    them before it launches.  Here the host writes such values into the
    scratch between two calls (no GPU fault involved), and the second call
    must still report no error and equal the workspace layout."""
    lib = abi.lib()
    w = workloads.WORKLOADS["prefill_cap"].scaled(4000)
    stream = torch.cuda.current_stream()
    inp = workloads.make_inputs(w, "cuda")
    plan = RoutePlan(_shape(w), "cuda")
    plan.gate(inp["logits"])
    gates_in = plan.gates.clone()
    plan.dispatch_layout()
    assert plan.status() == 0
    L2 = abi.Layout(w.T, w.E, w.k, w.P, w.capacity, "cuda")

    def call():
        g = gates_in.clone()
        rc = lib.moe_dispatch_layout_noalloc(
            ctypes.c_void_p(plan.topk_idx.data_ptr()), ctypes.c_void_p(plan.expert_counts.data_ptr()),
            w.T, w.E, w.k, w.P, w.capacity, ctypes.c_void_p(g.data_ptr()), ctypes.byref(L2.c),
            ctypes.c_void_p(stream.cuda_stream))
        assert rc == abi.MOE_OK
        assert lib.moe_get_status(ctypes.c_void_p(L2.c.ws), ctypes.c_void_p(stream.cuda_stream)) == 0
        R = int(plan.layout.offsets[w.E].item())
        for name in FIELDS:
            a, b = getattr(plan.layout, name), getattr(L2, name)
            if name == "src_pos":
                a, b = a[:R], b[:R]
            assert torch.equal(a, b), name
        assert torch.equal(plan.gates.view(torch.int32), g.view(torch.int32))

    call()
    # scratch header, 32-bit words: [0] status, [1] completed-tile counter,
    # [2] gate ticket, [3] test hook, [4] tile-id half and [5] epoch half of
    # the tile/epoch word; the per-partition token totals start at byte 1152
    words = torch.as_tensor(_DeviceWords(L2.c.ws, 1152 // 4 + w.P), device="cuda")
    words[1] = 5
    words[2] = 7
    words[4] = 3
    words[1152 // 4:] = 11
    torch.cuda.synchronize()
    call()
    call()
