"""Thin Python binding of libmoeroute's C ABI (include/moe_route.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, checks dtypes/devices/shapes of the torch tensors it is
given, passes their device pointers and the current CUDA stream, and raises
``MoeError`` on a non-zero status.  All routing work runs in the library's
CUDA kernels; there is no CPU fallback.  PyTorch only provides device memory
and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_DATA = 6

MOE_TOPK_SOFTMAX = 0
MOE_SOFTMAX_TOPK = 1

MOE_FP8_PER_TOKEN = 1
MOE_FP8_PER_EXPERT = 2
MOE_FP8_GLOBAL = 3

MOE_MAX_EXPERTS = 256
MOE_MAX_TOPK = 16
MOE_MAX_SHARED = 8
MOE_MAX_H_FP8 = 16384
MOE_NOALLOC_SCRATCH_BYTES = 2 << 20

_LIB = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class moe_layout(ctypes.Structure):
    """Mirror of ``struct moe_layout`` (host struct of device pointers)."""
    _fields_ = [
        ("T", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("P", ctypes.c_int32),
        ("capacity", ctypes.c_int32), ("r_max", ctypes.c_int32),
        ("ws", ctypes.c_void_p),
        ("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
        ("part_rows", ctypes.c_void_p), ("part_offsets", ctypes.c_void_p),
        ("part_tokens", ctypes.c_void_p), ("src_pos", ctypes.c_void_p),
        ("dst_row", ctypes.c_void_p), ("capacity_mask", ctypes.c_void_p),
        ("dropped", ctypes.c_void_p),
    ]


class moe_dedup(ctypes.Structure):
    """Mirror of ``struct moe_dedup`` (host struct of device pointers)."""
    _fields_ = [
        ("T", ctypes.c_int32), ("k", ctypes.c_int32), ("P", ctypes.c_int32), ("s_max", ctypes.c_int32),
        ("ws", ctypes.c_void_p),
        ("send_offsets", ctypes.c_void_p), ("send_row", ctypes.c_void_p), ("send_token", ctypes.c_void_p),
        ("slot_local", ctypes.c_void_p), ("slot_gate", ctypes.c_void_p),
    ]


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load libmoeroute.so.  Raises if it has not been built: the routing
    path has no substitute implementation."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.moe_workspace_size.argtypes = [I, I, I, I]
    L.moe_workspace_size.restype = SZ
    L.moe_workspace_init.argtypes = [P, SZ, P]
    L.moe_workspace_init.restype = I
    L.moe_rows_max.argtypes = [I, I, I, I]
    L.moe_rows_max.restype = ctypes.c_int64
    L.moe_gate.argtypes = [P, I, I, I, I, P, P, P, P, P, P, SZ, P]
    L.moe_gate.restype = I
    L.moe_route.argtypes = [P, I, I, I, I, I, I, P, P, P, P, P, ctypes.POINTER(moe_layout), P, SZ, P]
    L.moe_route.restype = I
    L.moe_route_launches.argtypes = [I, I, I, I, I]
    L.moe_route_launches.restype = I
    L.moe_dispatch_layout.argtypes = [P, P, I, I, I, I, I, P, ctypes.POINTER(moe_layout), P, SZ, P]
    L.moe_dispatch_layout.restype = I
    L.moe_dispatch_layout_reassign.argtypes = [P, P, I, I, I, I, I, P, ctypes.POINTER(moe_layout), P, SZ, P]
    L.moe_dispatch_layout_reassign.restype = I
    L.moe_dispatch_layout_noalloc.argtypes = [P, P, I, I, I, I, I, P, ctypes.POINTER(moe_layout), P]
    L.moe_dispatch_layout_noalloc.restype = I
    L.moe_dispatch.argtypes = [P, I, I, ctypes.POINTER(moe_layout), I, P, P, P]
    L.moe_dispatch.restype = I
    L.moe_combine.argtypes = [P, ctypes.POINTER(moe_layout), P, P, I, I, I, P, P]
    L.moe_combine.restype = I
    L.moe_quantize_rows.argtypes = [P, ctypes.POINTER(moe_layout), I, I, P, P, P]
    L.moe_quantize_rows.restype = I
    L.moe_combine_fp8.argtypes = [P, P, ctypes.POINTER(moe_layout), P, P, I, I, I, P, P]
    L.moe_combine_fp8.restype = I
    L.moe_combine_backward.argtypes = [P, P, ctypes.POINTER(moe_layout), P, I, I, P, P, P]
    L.moe_combine_backward.restype = I
    L.moe_dispatch_backward.argtypes = [P, ctypes.POINTER(moe_layout), I, I, P, P]
    L.moe_dispatch_backward.restype = I
    L.moe_gate_backward.argtypes = [P, P, P, I, I, I, I, P, P, SZ, P]
    L.moe_gate_backward.restype = I
    L.moe_dedup_scratch_size.argtypes = [I, I]
    L.moe_dedup_scratch_size.restype = SZ
    L.moe_dedup_layout.argtypes = [ctypes.POINTER(moe_layout), P, ctypes.POINTER(moe_dedup), P, SZ, P]
    L.moe_dedup_layout.restype = I
    L.moe_dispatch_dedup.argtypes = [P, I, I, ctypes.POINTER(moe_dedup), I, P, P, P]
    L.moe_dispatch_dedup.restype = I
    L.moe_combine_partials.argtypes = [P, ctypes.POINTER(moe_dedup), P, I, I, I, P, P]
    L.moe_combine_partials.restype = I
    L.moe_get_status.argtypes = [P, P]
    L.moe_get_status.restype = I
    L.moe_status_string.argtypes = [I]
    L.moe_status_string.restype = ctypes.c_char_p
    _LIB = L
    return L


def status_string(status: int) -> str:
    try:
        return lib().moe_status_string(int(status)).decode()
    except Exception:  # library not loadable: still describe the code
        return {0: "ok", 1: "invalid argument", 2: "unsupported size or option",
                3: "workspace too small", 4: "CUDA runtime error", 5: "device wait timed out",
                6: "invalid data found on the device"}.get(int(status), "unknown status")


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


# --------------------------------------------------------------------------
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------

def moe_workspace_size(T: int, E: int, k: int, P: int) -> int:
    return int(lib().moe_workspace_size(T, E, k, P))


def moe_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(lib().moe_workspace_init(_ptr(ws, name="ws"), _nbytes(ws), _stream(stream)),
           "moe_workspace_init")


def moe_rows_max(T: int, E: int, k: int, capacity: int) -> int:
    return int(lib().moe_rows_max(T, E, k, capacity))


def moe_gate(logits, k: int, mode: int, topk_idx, gates, expert_counts, aux_loss, entropy, ws,
             stream=None) -> None:
    T, E = logits.shape
    _check(lib().moe_gate(_ptr(logits, torch.float32, "logits"), T, E, k, mode,
                          _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(gates, torch.float32, "gates"),
                          _ptr(expert_counts, torch.int32, "expert_counts"),
                          _ptr(aux_loss, torch.float64, "aux_loss"),
                          _ptr(entropy, torch.float64, "entropy"),
                          _ptr(ws, name="ws"), _nbytes(ws), _stream(stream)), "moe_gate")


def moe_route(logits, k: int, mode: int, P: int, capacity: int, topk_idx, gates, expert_counts, aux_loss, entropy,
              layout: "Layout", ws, stream=None) -> None:
    """moe_gate + moe_dispatch_layout, in one launch where the batch allows
    (moe_route_launches)."""
    T, E = logits.shape
    _check_layout_fits(layout, T, E, k, P, capacity, "moe_route")
    _check(lib().moe_route(_ptr(logits, torch.float32, "logits"), T, E, k, mode, P, capacity,
                           _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(gates, torch.float32, "gates"),
                           _ptr(expert_counts, torch.int32, "expert_counts"),
                           _ptr(aux_loss, torch.float64, "aux_loss"), _ptr(entropy, torch.float64, "entropy"),
                           ctypes.byref(layout.c), _ptr(ws, name="ws"), _nbytes(ws), _stream(stream)), "moe_route")


def moe_route_launches(T: int, E: int, k: int, mode: int, P: int) -> int:
    """Kernel launches moe_route takes for these sizes on the current device
    (1 fused, 2 gate + layout, 0 unsupported)."""
    return int(lib().moe_route_launches(T, E, k, mode, P))


def _check_layout_fits(layout: "Layout", T: int, E: int, k: int, P: int, capacity: int, where: str):
    """Refuse, before the foreign call, a layout call whose sizes exceed the
    buffers `layout` was allocated for: the kernel writes T*k entries of
    dst_row / capacity_mask and up to moe_rows_max rows of src_pos."""
    if E > layout.E or P > layout.P:
        raise ValueError(f"{where}: layout allocated for E={layout.E}, P={layout.P}, called with E={E}, P={P}")
    if T < 0 or T * k > layout.A:
        raise ValueError(f"{where}: T*k = {T * k} assignments, the layout holds {layout.A}")
    r = moe_rows_max(T, E, k, capacity)
    if r > layout.r_max:
        raise ValueError(f"{where}: up to {r} packed rows for T={T}, k={k}, capacity={capacity}; "
                         f"the layout holds {layout.r_max}")


def moe_dispatch_layout(topk_idx, expert_counts, T: int, E: int, k: int, P: int, capacity: int,
                        gates_or_null, layout: "Layout", ws, stream=None) -> None:
    _check_layout_fits(layout, T, E, k, P, capacity, "moe_dispatch_layout")
    _check(lib().moe_dispatch_layout(_ptr(topk_idx, torch.int32, "topk_idx"),
                                     _ptr(expert_counts, torch.int32, "expert_counts"),
                                     T, E, k, P, capacity,
                                     _ptr(gates_or_null, torch.float32, "gates"),
                                     ctypes.byref(layout.c), _ptr(ws, name="ws"), _nbytes(ws),
                                     _stream(stream)), "moe_dispatch_layout")


def moe_dispatch_layout_reassign(topk_idx, expert_counts, T: int, E: int, k: int, P: int, capacity: int,
                                 gates_or_null, layout: "Layout", ws, stream=None) -> None:
    _check_layout_fits(layout, T, E, k, P, capacity, "moe_dispatch_layout_reassign")
    _check(lib().moe_dispatch_layout_reassign(_ptr(topk_idx, torch.int32, "topk_idx"),
                                              _ptr(expert_counts, torch.int32, "expert_counts"),
                                              T, E, k, P, capacity,
                                              _ptr(gates_or_null, torch.float32, "gates"),
                                              ctypes.byref(layout.c), _ptr(ws, name="ws"), _nbytes(ws),
                                              _stream(stream)), "moe_dispatch_layout_reassign")


def moe_dispatch_layout_noalloc(topk_idx, expert_counts, T: int, E: int, k: int, P: int,
                                capacity: int, gates_or_null, layout: "Layout", stream=None) -> None:
    """moe_dispatch_layout without a workspace argument: the library's own
    fixed scratch is used (no device allocation anywhere in the call)."""
    _check_layout_fits(layout, T, E, k, P, capacity, "moe_dispatch_layout_noalloc")
    _check(lib().moe_dispatch_layout_noalloc(_ptr(topk_idx, torch.int32, "topk_idx"),
                                             _ptr(expert_counts, torch.int32, "expert_counts"),
                                             T, E, k, P, capacity,
                                             _ptr(gates_or_null, torch.float32, "gates"),
                                             ctypes.byref(layout.c), _stream(stream)),
           "moe_dispatch_layout_noalloc")


def _check_rows(t, rows: int, name: str, where: str):
    """A row buffer read or written up to `rows` rows must hold them."""
    if t is not None and t.shape[0] < rows:
        raise ValueError(f"{where}: {name} has {t.shape[0]} rows, needs {rows}")


def moe_dispatch(x, T: int, H: int, layout: "Layout", fp8: int, packed, scales=None,
                 stream=None) -> None:
    _check_rows(x, T, "x", "moe_dispatch")
    _check_rows(packed, layout.c.r_max, "packed", "moe_dispatch")
    _check_rows(scales, layout.c.r_max, "scales", "moe_dispatch")
    _check(lib().moe_dispatch(_ptr(x, torch.bfloat16, "x"), T, H, ctypes.byref(layout.c), int(fp8),
                              _ptr(packed, torch.uint8 if fp8 else torch.bfloat16, "packed"),
                              _ptr(scales, torch.float32, "scales"), _stream(stream)), "moe_dispatch")


def moe_combine(expert_out, layout: "Layout", gates, shared_out, Ks: int, T: int, H: int, y,
                stream=None) -> None:
    _check_rows(expert_out, layout.c.r_max, "expert_out", "moe_combine")
    _check_rows(y, T, "y", "moe_combine")
    _check(lib().moe_combine(_ptr(expert_out, torch.bfloat16, "expert_out"), ctypes.byref(layout.c),
                             _ptr(gates, torch.float32, "gates"),
                             _ptr(shared_out, torch.bfloat16, "shared_out"), Ks, T, H,
                             _ptr(y, torch.bfloat16, "y"), _stream(stream)), "moe_combine")


def moe_quantize_rows(rows, layout: "Layout", H: int, mode: int, codes, scales, stream=None) -> None:
    for t, name in ((rows, "rows"), (codes, "codes"), (scales, "scales")):
        _check_rows(t, layout.c.r_max, name, "moe_quantize_rows")
    _check(lib().moe_quantize_rows(_ptr(rows, torch.bfloat16, "rows"), ctypes.byref(layout.c), H, int(mode),
                                   _ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"),
                                   _stream(stream)), "moe_quantize_rows")


def moe_combine_fp8(codes, scales, layout: "Layout", gates, shared_out, Ks: int, T: int, H: int, y,
                    stream=None) -> None:
    _check_rows(codes, layout.c.r_max, "codes", "moe_combine_fp8")
    _check_rows(scales, layout.c.r_max, "scales", "moe_combine_fp8")
    _check_rows(y, T, "y", "moe_combine_fp8")
    _check(lib().moe_combine_fp8(_ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"),
                                 ctypes.byref(layout.c), _ptr(gates, torch.float32, "gates"),
                                 _ptr(shared_out, torch.bfloat16, "shared_out"), Ks, T, H,
                                 _ptr(y, torch.bfloat16, "y"), _stream(stream)), "moe_combine_fp8")


def moe_combine_backward(dy, expert_out, layout: "Layout", gates, T: int, H: int, d_expert_out, d_gates,
                         stream=None) -> None:
    _check_rows(expert_out, layout.c.r_max, "expert_out", "moe_combine_backward")
    _check_rows(d_expert_out, layout.c.r_max, "d_expert_out", "moe_combine_backward")
    _check_rows(dy, T, "dy", "moe_combine_backward")
    _check(lib().moe_combine_backward(_ptr(dy, torch.bfloat16, "dy"),
                                      _ptr(expert_out, torch.bfloat16, "expert_out"), ctypes.byref(layout.c),
                                      _ptr(gates, torch.float32, "gates"), T, H,
                                      _ptr(d_expert_out, torch.bfloat16, "d_expert_out"),
                                      _ptr(d_gates, torch.float32, "d_gates"), _stream(stream)),
           "moe_combine_backward")


def moe_dispatch_backward(d_packed, layout: "Layout", T: int, H: int, dx, stream=None) -> None:
    _check_rows(d_packed, layout.c.r_max, "d_packed", "moe_dispatch_backward")
    _check_rows(dx, T, "dx", "moe_dispatch_backward")
    _check(lib().moe_dispatch_backward(_ptr(d_packed, torch.bfloat16, "d_packed"), ctypes.byref(layout.c), T, H,
                                       _ptr(dx, torch.bfloat16, "dx"), _stream(stream)), "moe_dispatch_backward")


def moe_gate_backward(logits, topk_idx, d_gates, mode: int, d_logits, ws, stream=None) -> None:
    T, E = logits.shape
    k = topk_idx.shape[1]
    _check(lib().moe_gate_backward(_ptr(logits, torch.float32, "logits"), _ptr(topk_idx, torch.int32, "topk_idx"),
                                   _ptr(d_gates, torch.float32, "d_gates"), T, E, k, mode,
                                   _ptr(d_logits, torch.float32, "d_logits"), _ptr(ws, name="ws"), _nbytes(ws),
                                   _stream(stream)), "moe_gate_backward")


def moe_dedup_scratch_size(T: int, P: int) -> int:
    return int(lib().moe_dedup_scratch_size(T, P))


def moe_dedup_layout(layout: "Layout", gates, dedup: "Dedup", stream=None, groups: int | None = None) -> None:
    """Send rows of `layout` per partition, or, with `groups`, per group of
    E/groups consecutive experts (e.g. one group per rank of an
    expert-parallel exchange whose ranks own several partitions): the call
    then sees a copy of the layout struct with P = groups."""
    c = layout.c
    if groups is not None and groups != c.P:
        if groups < 1 or layout.E % groups != 0:
            raise ValueError(f"groups must divide E = {layout.E}")
        c = moe_layout.from_buffer_copy(layout.c)
        c.P = groups
    if dedup.P != c.P or dedup.T < c.T or dedup.k != c.k:
        raise ValueError(f"moe_dedup_layout: the send-row buffers hold T={dedup.T}, k={dedup.k}, P={dedup.P}; "
                         f"the call has T={c.T}, k={c.k}, P={c.P}")
    _check(lib().moe_dedup_layout(ctypes.byref(c), _ptr(gates, torch.float32, "gates"), ctypes.byref(dedup.c),
                                  _ptr(dedup.scratch, name="scratch"), _nbytes(dedup.scratch), _stream(stream)),
           "moe_dedup_layout")


def moe_dispatch_dedup(x, T: int, H: int, dedup: "Dedup", fp8: int, send_buf, scales=None, stream=None) -> None:
    _check(lib().moe_dispatch_dedup(_ptr(x, torch.bfloat16, "x"), T, H, ctypes.byref(dedup.c), int(fp8),
                                    _ptr(send_buf, torch.uint8 if fp8 else torch.bfloat16, "send_buf"),
                                    _ptr(scales, torch.float32, "scales"), _stream(stream)), "moe_dispatch_dedup")


def moe_combine_partials(partials, dedup: "Dedup", shared_out, Ks: int, T: int, H: int, y, stream=None) -> None:
    _check(lib().moe_combine_partials(_ptr(partials, torch.bfloat16, "partials"), ctypes.byref(dedup.c),
                                      _ptr(shared_out, torch.bfloat16, "shared_out"), Ks, T, H,
                                      _ptr(y, torch.bfloat16, "y"), _stream(stream)), "moe_combine_partials")


def moe_get_status(ws, stream=None) -> int:
    """Synchronise, return and clear the device status recorded in ``ws``."""
    return int(lib().moe_get_status(_ptr(ws, name="ws"), _stream(stream)))


# --------------------------------------------------------------------------
# buffer helpers (allocation through PyTorch)
# --------------------------------------------------------------------------

class Layout:
    """Device buffers of one ``moe_layout`` plus the ctypes struct that
    points at them."""

    def __init__(self, T: int, E: int, k: int, P: int, capacity: int = 0, device="cuda"):
        r_max = moe_rows_max(T, E, k, capacity)
        if r_max < 0:
            raise MoeError(MOE_ERR_UNSUPPORTED, "Layout")
        i32 = dict(dtype=torch.int32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.part_rows = torch.empty(P, **i32)
        self.part_offsets = torch.empty(P + 1, **i32)
        self.part_tokens = torch.empty(P, **i32)
        self.src_pos = torch.empty(max(r_max, 1), **i32)
        self.dst_row = torch.empty(max(T * k, 1), **i32)
        self.capacity_mask = torch.empty(max(T * k, 1), dtype=torch.uint8, device=device)
        self.dropped = torch.empty(1, dtype=torch.int64, device=device)
        # the sizes the buffers hold: a layout call must not exceed them
        self.T, self.E, self.k, self.P, self.capacity = T, E, k, P, capacity
        self.A = T * k
        self.r_max = r_max
        c = moe_layout()
        for name in ("counts", "offsets", "part_rows", "part_offsets", "part_tokens", "src_pos",
                     "dst_row", "capacity_mask", "dropped"):
            setattr(c, name, getattr(self, name).data_ptr())
        self.c = c


class Dedup:
    """Device buffers of one ``moe_dedup`` (send rows of T tokens over P
    partitions) plus its scratch and the ctypes struct."""

    def __init__(self, T: int, k: int, P: int, device="cuda"):
        s_max = max(T * min(k, P), 1)
        i32 = dict(dtype=torch.int32, device=device)
        self.send_offsets = torch.empty(P + 1, **i32)
        self.send_row = torch.empty((max(T, 1), P), **i32)
        self.send_token = torch.empty(s_max, **i32)
        self.slot_local = torch.empty((s_max, k), **i32)
        self.slot_gate = torch.empty((s_max, k), dtype=torch.float32, device=device)
        n = moe_dedup_scratch_size(T, P)
        if n == 0:
            raise MoeError(MOE_ERR_UNSUPPORTED, "moe_dedup_scratch_size")
        self.scratch = torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=device)
        self.s_max = s_max
        self.T, self.k, self.P = T, k, P
        c = moe_dedup()
        for name in ("send_offsets", "send_row", "send_token", "slot_local", "slot_gate"):
            setattr(c, name, getattr(self, name).data_ptr())
        self.c = c


def alloc_workspace(T: int, E: int, k: int, P: int, device="cuda", stream=None) -> torch.Tensor:
    n = moe_workspace_size(T, E, k, P)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED, "moe_workspace_size")
    ws = torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws
