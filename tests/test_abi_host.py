"""CPU-only checks of the C-ABI library: it builds, loads, exports every
entry point include/moe_route.h declares, and its host-side size queries
and argument checks behave as documented (no CUDA call is reached)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    from combine_moe_gate_warp_gb300 import abi
    return abi.lib()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"moe_gate", "moe_dispatch_layout", "moe_dispatch", "moe_combine", "moe_get_status",
            "moe_workspace_size", "moe_workspace_init", "moe_rows_max", "moe_status_string",
            "moe_combine_backward", "moe_dispatch_backward", "moe_gate_backward", "moe_quantize_rows",
            "moe_combine_fp8", "moe_dispatch_layout_reassign", "moe_dedup_scratch_size", "moe_dedup_layout",
            "moe_dispatch_dedup", "moe_combine_partials"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def test_workspace_and_rows_queries(lib):
    from combine_moe_gate_warp_gb300 import abi
    # 8 KiB of counters, one 8-byte look-back flag word per (layout tile,
    # expert) (tiles of 1024..8192 assignments), then one 4-byte histogram
    # word per (moe_route tile, expert) (tiles of >= 32 tokens, at most 1024)
    assert abi.moe_workspace_size(16384, 16, 2, 4) == 8192 + 32 * 16 * 8 + 512 * 16 * 4
    assert abi.moe_workspace_size(262144, 64, 8, 8) == 8192 + 256 * 64 * 8 + 1024 * 64 * 4
    assert abi.moe_workspace_size(2048, 16, 8, 4) == 8192 + 16 * 16 * 8 + 64 * 16 * 4
    assert abi.moe_workspace_size(100, 16, 2, 4) == 8192 + 1 * 16 * 8 + 4 * 16 * 4
    assert abi.moe_workspace_size(1000, 8, 16, 4) == 8192 + 16 * 8 * 8 + 32 * 8 * 4
    assert abi.moe_workspace_size(100, 16, 2, 3) == 0   # P does not divide E
    assert abi.moe_workspace_size(100, 300, 2, 4) == 0  # E too large
    assert abi.moe_rows_max(262144, 64, 8, 40960) == 2097152
    assert abi.moe_rows_max(100, 8, 2, 5) == 40
    assert abi.moe_rows_max(100, 8, 2, 0) == 200
    assert abi.moe_rows_max(100, 8, 17, 0) == -1        # k > 16
    assert abi.moe_rows_max(100, 8, 9, 0) == 900        # k > E: rows with empty slots


def test_argument_checks_return_before_any_cuda_call(lib):
    from combine_moe_gate_warp_gb300 import abi
    P = ctypes.c_void_p
    fake = P(1 << 20)
    # k = 0, E too large, mode invalid, T < 0
    assert lib.moe_gate(fake, 10, 8, 0, 0, fake, fake, fake, fake, fake, fake, 1 << 20, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_gate(fake, 10, 300, 2, 0, fake, fake, fake, fake, fake, fake, 1 << 20, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_gate(fake, 10, 8, 2, 9, fake, fake, fake, fake, fake, fake, 1 << 20, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_gate(fake, -1, 8, 2, 0, fake, fake, fake, fake, fake, fake, 1 << 20, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_gate(P((1 << 20) + 4), 10, 8, 2, 0, fake, fake, fake, fake, fake, fake, 1 << 20, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_gate(fake, 10, 8, 2, 0, fake, fake, fake, fake, fake, fake, 100, None) == abi.MOE_ERR_WORKSPACE_TOO_SMALL
    L = abi.moe_layout()
    assert lib.moe_dispatch_layout(fake, fake, 10, 8, 2, 3, 0, None, ctypes.byref(L), fake, 1 << 20, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_dispatch_layout(fake, fake, 10, 8, 2, 4, 0, None, ctypes.byref(L), fake, 1 << 20, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_layout_reassign(fake, fake, 10, 8, 2, 3, 5, None, ctypes.byref(L), fake, 1 << 20,
                                            None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_dispatch(fake, 10, 64, None, 0, fake, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(fake, 10, 64, None, 4, fake, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_rows(fake, None, 64, 1, fake, fake, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_fp8(fake, fake, None, fake, None, 0, 10, 64, fake, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(fake, None, fake, None, 0, 10, 64, fake, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_backward(fake, fake, None, fake, 10, 64, fake, fake, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_backward(fake, None, 10, 64, fake, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_backward(fake, fake, fake, 10, 8, 2, 0, fake, fake, 100, None) == abi.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_gate_backward(fake, fake, fake, 10, 8, 2, 7, fake, fake, 1 << 20, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_backward(fake, fake, fake, 10, 8, 9, 0, fake, fake, 1 << 20, None) == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_dedup_scratch_size(100, 17) == 0 and lib.moe_dedup_scratch_size(100, 8) > 0
    assert lib.moe_dedup_layout(None, fake, None, fake, 1 << 20, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_dedup(fake, 10, 64, None, 0, fake, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_partials(fake, None, None, 0, 10, 64, fake, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_get_status(None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_status_string(5) == b"device wait timed out"


def test_binding_names_match_the_c_abi():
    from combine_moe_gate_warp_gb300 import abi
    for n in ("moe_gate", "moe_dispatch_layout", "moe_dispatch", "moe_combine", "moe_get_status",
              "moe_workspace_size", "moe_workspace_init", "moe_rows_max", "moe_combine_backward",
              "moe_dispatch_backward", "moe_gate_backward", "moe_quantize_rows", "moe_combine_fp8",
              "moe_dispatch_layout_reassign", "moe_dedup_scratch_size", "moe_dedup_layout", "moe_dispatch_dedup",
              "moe_combine_partials"):
        assert callable(getattr(abi, n))
    # the struct mirrors the header's field order
    hdr = open(os.path.join(ROOT, "include", "moe_route.h")).read()
    body = hdr[hdr.index("typedef struct moe_layout {"):hdr.index("} moe_layout;")]
    fields = re.findall(r"\*?(\w+)(?:,|;)", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
    assert [f for f, _ in abi.moe_layout._fields_] == fields


def test_layout_wrappers_refuse_sizes_beyond_the_layout(lib):
    """The binding refuses, before the foreign call, a layout call that would
    write past the buffers the Layout was allocated for: more assignments
    (T*k), more packed rows (capacity removed or raised), or another E / P."""
    import torch

    from combine_moe_gate_warp_gb300 import abi
    lay = abi.Layout(100, 8, 2, 4, capacity=10, device="cpu")  # r_max = min(200, 8 * 10) = 80
    assert lay.r_max == 80 and lay.A == 200
    ids = torch.zeros((300, 2), dtype=torch.int32)
    cnt = torch.zeros(8, dtype=torch.int32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    for fn in (abi.moe_dispatch_layout, abi.moe_dispatch_layout_reassign):
        with pytest.raises(ValueError, match="assignments"):
            fn(ids, cnt, 150, 8, 2, 4, 10, None, lay, ws)
        with pytest.raises(ValueError, match="packed rows"):
            fn(ids, cnt, 100, 8, 2, 4, 0, None, lay, ws)      # no capacity: up to 200 rows
        with pytest.raises(ValueError, match="packed rows"):
            fn(ids, cnt, 100, 8, 2, 4, 11, None, lay, ws)
        with pytest.raises(ValueError, match="E=8, P=4"):
            fn(ids, cnt, 100, 8, 2, 8, 10, None, lay, ws)     # more partitions than allocated
        with pytest.raises(ValueError, match="E=8, P=4"):
            fn(ids, cnt, 100, 16, 2, 4, 10, None, lay, ws)    # more experts than allocated
    with pytest.raises(ValueError, match="packed rows"):
        abi.moe_dispatch_layout_noalloc(ids, cnt, 100, 8, 2, 4, 0, None, lay)
    # the sizes it was built for pass the check (and stop at the CPU tensors)
    with pytest.raises(ValueError, match="CUDA tensor"):
        abi.moe_dispatch_layout(ids, cnt, 100, 8, 2, 4, 10, None, lay, ws)
    with pytest.raises(ValueError, match="CUDA tensor"):
        abi.moe_dispatch_layout(ids, cnt, 40, 8, 2, 4, 0, None, lay, ws)  # fewer tokens, no capacity: 80 rows
    # consumers: packed-row buffers must hold the layout's r_max rows
    lay.c.r_max = 80
    short = torch.zeros((79, 16), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="expert_out has 79 rows"):
        abi.moe_combine(short, lay, None, None, 0, 100, 16, torch.zeros((100, 16), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="packed has 79 rows"):
        abi.moe_dispatch(torch.zeros((100, 16), dtype=torch.bfloat16), 100, 16, lay, 0, short)
    with pytest.raises(ValueError, match="d_packed has 79 rows"):
        abi.moe_dispatch_backward(short, lay, 100, 16, torch.zeros((100, 16), dtype=torch.bfloat16))


def test_route_plan_requires_r_max_rows():
    """RoutePlan's combine, quantise and backward calls read packed-row
    tensors up to R, which only the device knows: fewer than r_max rows are
    refused on the host."""
    import torch

    from combine_moe_gate_warp_gb300.pipeline import _check_packed_rows
    with pytest.raises(ValueError, match="r_max = 80"):
        _check_packed_rows(torch.zeros((79, 16), dtype=torch.bfloat16), torch.bfloat16, 80, 16, "expert_out")
    with pytest.raises(ValueError, match=r"\[rows, 16\]"):
        _check_packed_rows(torch.zeros((80, 8), dtype=torch.bfloat16), torch.bfloat16, 80, 16, "expert_out")
    with pytest.raises(ValueError, match="CUDA tensor"):  # enough rows: only the device check remains
        _check_packed_rows(torch.zeros((80, 16), dtype=torch.bfloat16), torch.bfloat16, 80, 16, "expert_out")
