"""CPU oracle for MoE token routing -- TEST INFRASTRUCTURE ONLY.

A ctypes binding over ``moe_oracle.c`` (plain C, single-threaded, fp64 where
the definition allows).  The test suite, the smoke check and the benchmark's
CPU-baseline / reference arm are the only callers.  The CUDA library never
imports, links or executes anything here, and this module shares no code
with it.

Every wrapper takes and returns numpy arrays (bf16 tensors travel as their
uint16 bit patterns).  The C functions cite the source passages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_LIB = None

_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source with gcc (no -ffast-math)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _LIB
    if _LIB is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.oracle_topk.argtypes = [P, I64, I, I, P]
        lib.oracle_topk.restype = I
        lib.oracle_gates.argtypes = [P, P, I64, I, I, I, P]
        lib.oracle_gates.restype = I
        lib.oracle_stats.argtypes = [P, I64, I, I, P, P, P]
        lib.oracle_stats.restype = I
        lib.oracle_layout.argtypes = [P, I64, I, I, I, I64, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_layout.restype = I
        lib.oracle_dispatch_bf16_rows.argtypes = [P, I64, I, P, P, I64, P]
        lib.oracle_dispatch_bf16_rows.restype = None
        lib.oracle_e4m3_satfinite.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_satfinite.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_quantize_row_fp8.argtypes = [P, I64, P, P, P]
        lib.oracle_quantize_row_fp8.restype = None
        lib.oracle_dispatch_fp8_rows.argtypes = [P, I64, I, P, P, I64, P, P]
        lib.oracle_dispatch_fp8_rows.restype = None
        lib.oracle_combine_f32order_tokens.argtypes = [P, I64, I, P, P, P, I, I64, P, I64, P]
        lib.oracle_combine_f32order_tokens.restype = None
        lib.oracle_combine_ref64_tokens.argtypes = [P, I64, I, P, P, P, I, I64, P, I64, P, P]
        lib.oracle_combine_ref64_tokens.restype = None
        lib.oracle_layout_reassign.argtypes = [P, I64, I, I, I, I64, P, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_layout_reassign.restype = I
        lib.oracle_dedup_layout.argtypes = [P, P, P, I64, I, I, I, P, P, P, P, P]
        lib.oracle_dedup_layout.restype = I64
        lib.oracle_fp8_group_params.argtypes = [P, I64, P, P, I64, I64, P]
        lib.oracle_fp8_group_params.restype = I
        lib.oracle_quantize_rows_with_params.argtypes = [P, I64, P, P, I64, P, P, P]
        lib.oracle_quantize_rows_with_params.restype = None
        lib.oracle_combine_fp8_f32order_tokens.argtypes = [P, P, I64, I, P, P, P, I, I64, P, I64, P]
        lib.oracle_combine_fp8_f32order_tokens.restype = None
        lib.oracle_combine_fp8_ref64_tokens.argtypes = [P, P, I64, I, P, P, P, I, I64, P, I64, P, P]
        lib.oracle_combine_fp8_ref64_tokens.restype = None
        lib.oracle_combine_backward_tokens.argtypes = [P, P, I64, I, P, P, P, I64, P, P]
        lib.oracle_combine_backward_tokens.restype = None
        lib.oracle_dispatch_backward_tokens.argtypes = [P, I64, I, P, P, I64, P, P]
        lib.oracle_dispatch_backward_tokens.restype = None
        lib.oracle_gate_backward.argtypes = [P, P, P, I64, I, I, I, P]
        lib.oracle_gate_backward.restype = I
        lib.oracle_bf16_from_float.argtypes = [ctypes.c_float]
        lib.oracle_bf16_from_float.restype = ctypes.c_uint16
        _LIB = lib
    return _LIB


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


TOPK_SOFTMAX = 0
SOFTMAX_TOPK = 1


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Top-k expert ids per token, int32 [T, k] (value desc, ties to lower id)."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    rc = _lib().oracle_topk(_p(logits), T, E, k, _p(out))
    if rc != 0:
        raise ValueError(f"oracle_topk failed ({rc}): logits must be finite")
    return out


def gates(logits: np.ndarray, topk_idx: np.ndarray, mode: int) -> np.ndarray:
    """Gate weights in fp64 [T, k]."""
    logits = _c(logits, np.float32)
    topk_idx = _c(topk_idx, np.int32)
    T, E = logits.shape
    k = topk_idx.shape[1]
    out = np.empty((T, k), np.float64)
    rc = _lib().oracle_gates(_p(logits), _p(topk_idx), T, E, k, mode, _p(out))
    if rc != 0:
        raise ValueError("bad gate mode")
    return out


def stats(topk_idx: np.ndarray, E: int):
    """(expert_counts int32 [E], aux_loss float, entropy float)."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, np.int32)
    aux = np.zeros(1, np.float64)
    ent = np.zeros(1, np.float64)
    rc = _lib().oracle_stats(_p(topk_idx), T, E, k, _p(counts), _p(aux), _p(ent))
    if rc != 0:
        raise ValueError("expert id out of range")
    return counts, float(aux[0]), float(ent[0])


def gate(logits: np.ndarray, k: int, mode: int):
    """The whole gate step: (topk_idx, gates fp64, counts, aux, entropy)."""
    idx = topk(logits, k)
    g = gates(logits, idx, mode)
    counts, aux, ent = stats(idx, logits.shape[1])
    return idx, g, counts, aux, ent


def layout(topk_idx: np.ndarray, E: int, P: int, capacity: int = 0, gates_f32=None):
    """Dispatch layout.  Returns a dict of numpy arrays; ``gates_f32`` (if
    given, float32 [T, k]) is copied and zeroed where dropped."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    A = T * k
    r_max = A if capacity <= 0 else min(A, E * capacity)
    g = None if gates_f32 is None else np.array(gates_f32, dtype=np.float32, copy=True, order="C")
    out = dict(
        counts=np.empty(E, np.int32),
        offsets=np.empty(E + 1, np.int32),
        dst_row=np.empty(A, np.int32),
        src_pos=np.full(max(r_max, 1), -7, np.int32),
        capacity_mask=np.empty(max(A, 1), np.uint8),
        part_rows=np.empty(P, np.int32),
        part_offsets=np.empty(P + 1, np.int32),
        part_tokens=np.empty(P, np.int32),
    )
    dropped = np.zeros(1, np.int64)
    rc = _lib().oracle_layout(
        _p(topk_idx), T, E, k, P, capacity, _p(g),
        _p(out["counts"]), _p(out["offsets"]), _p(out["dst_row"]), _p(out["src_pos"]),
        _p(out["capacity_mask"]), _p(out["part_rows"]), _p(out["part_offsets"]),
        _p(out["part_tokens"]), _p(dropped))
    if rc != 0:
        raise ValueError(f"oracle_layout failed ({rc})")
    R = int(out["offsets"][E])
    out["src_pos"] = out["src_pos"][:R]
    out["capacity_mask"] = out["capacity_mask"][:A]
    out["dropped"] = int(dropped[0])
    out["R"] = R
    if g is not None:
        out["gates"] = g
    return out


def layout_reassign(topk_idx: np.ndarray, E: int, P: int, capacity: int, gates_f32=None):
    """Dispatch layout with capacity overflow re-assigned to the least-loaded
    expert (capacity > 0).  Same keys as ``layout`` plus ``final_expert``;
    capacity_mask is 1 kept, 2 re-assigned, 0 dropped."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    A = T * k
    r_max = min(A, E * capacity)
    g = None if gates_f32 is None else np.array(gates_f32, dtype=np.float32, copy=True, order="C")
    out = dict(
        counts=np.empty(E, np.int32),
        offsets=np.empty(E + 1, np.int32),
        dst_row=np.empty(max(A, 1), np.int32),
        src_pos=np.full(max(r_max, 1), -7, np.int32),
        capacity_mask=np.empty(max(A, 1), np.uint8),
        final_expert=np.empty(max(A, 1), np.int32),
        part_rows=np.empty(P, np.int32),
        part_offsets=np.empty(P + 1, np.int32),
        part_tokens=np.empty(P, np.int32),
    )
    dropped = np.zeros(1, np.int64)
    rc = _lib().oracle_layout_reassign(
        _p(topk_idx), T, E, k, P, capacity, _p(g),
        _p(out["counts"]), _p(out["offsets"]), _p(out["dst_row"]), _p(out["src_pos"]),
        _p(out["capacity_mask"]), _p(out["final_expert"]), _p(out["part_rows"]), _p(out["part_offsets"]),
        _p(out["part_tokens"]), _p(dropped))
    if rc != 0:
        raise ValueError(f"oracle_layout_reassign failed ({rc})")
    R = int(out["offsets"][E])
    for key in ("dst_row", "capacity_mask", "final_expert"):
        out[key] = out[key][:A]
    out["src_pos"] = out["src_pos"][:R]
    out["dropped"] = int(dropped[0])
    out["R"] = R
    if g is not None:
        out["gates"] = g
    return out


def dedup_layout(dst_row, offsets, gates_f32, T: int, E: int, k: int, P: int):
    """Per-partition token de-duplication of a layout (see the C function).
    Returns dict(send_offsets [P+1], send_row [T, P], send_token [S],
    slot_local [S, k], slot_gate [S, k], S)."""
    dst_row = _c(dst_row, np.int32)
    offsets = _c(offsets, np.int32)
    gates_f32 = _c(gates_f32, np.float32)
    s_max = max(T * min(k, P), 1)
    out = dict(send_offsets=np.empty(P + 1, np.int32), send_row=np.empty((max(T, 1), P), np.int32),
               send_token=np.empty(s_max, np.int32), slot_local=np.empty((s_max, k), np.int32),
               slot_gate=np.empty((s_max, k), np.float32))
    S = _lib().oracle_dedup_layout(_p(dst_row), _p(offsets), _p(gates_f32), T, E, k, P, _p(out["send_offsets"]),
                                   _p(out["send_row"]), _p(out["send_token"]), _p(out["slot_local"]),
                                   _p(out["slot_gate"]))
    if S < 0:
        raise ValueError("oracle_dedup_layout failed")
    out["S"] = int(S)
    out["send_row"] = out["send_row"][:T]
    for key in ("send_token", "slot_local", "slot_gate"):
        out[key] = out[key][:S]
    return out


def dispatch_bf16_rows(x_bits: np.ndarray, k: int, src_pos: np.ndarray, rows) -> np.ndarray:
    """Packed bf16 rows (uint16 bit patterns) for the listed packed-row ids."""
    x_bits = _c(x_bits, np.uint16)
    src_pos = _c(src_pos, np.int32)
    rows = _c(rows, np.int64)
    H = x_bits.shape[1]
    out = np.empty((rows.size, H), np.uint16)
    _lib().oracle_dispatch_bf16_rows(_p(x_bits), H, k, _p(src_pos), _p(rows), rows.size, _p(out))
    return out


def e4m3(v: float) -> int:
    return int(_lib().oracle_e4m3_satfinite(float(v)))


def e4m3_array(v: np.ndarray) -> np.ndarray:
    """Element-wise e4m3 satfinite RNE encode of float32 values."""
    f = _lib().oracle_e4m3_satfinite
    flat = _c(v, np.float32).ravel()
    return np.fromiter((f(float(a)) for a in flat), dtype=np.uint8, count=flat.size).reshape(np.shape(v))


def e4m3_decode(c: int) -> float:
    return float(_lib().oracle_e4m3_decode(int(c)))


def quantize_row_fp8(xrow_bits: np.ndarray):
    """(codes uint8 [H], scale, zero) for one token row."""
    xrow_bits = _c(xrow_bits, np.uint16)
    H = xrow_bits.size
    codes = np.empty(H, np.uint8)
    s = np.zeros(1, np.float32)
    z = np.zeros(1, np.float32)
    _lib().oracle_quantize_row_fp8(_p(xrow_bits), H, _p(codes), _p(s), _p(z))
    return codes, float(s[0]), float(z[0])


def dispatch_fp8_rows(x_bits: np.ndarray, k: int, src_pos: np.ndarray, rows):
    """(codes uint8 [n, H], scales float32 [n, 2]) for the listed rows."""
    x_bits = _c(x_bits, np.uint16)
    src_pos = _c(src_pos, np.int32)
    rows = _c(rows, np.int64)
    H = x_bits.shape[1]
    codes = np.empty((rows.size, H), np.uint8)
    scales = np.empty((rows.size, 2), np.float32)
    _lib().oracle_dispatch_fp8_rows(_p(x_bits), H, k, _p(src_pos), _p(rows), rows.size,
                                    _p(codes), _p(scales))
    return codes, scales


FP8_PER_TOKEN, FP8_PER_EXPERT, FP8_GLOBAL = 1, 2, 3


def fp8_group_params(src_bits, src_row, group, ngroups):
    """(scale, zero) float32 [ngroups, 2] over the rows of each group."""
    src_bits = _c(src_bits, np.uint16)
    src_row = _c(src_row, np.int64)
    group = _c(group, np.int32)
    params = np.empty((max(int(ngroups), 1), 2), np.float32)
    rc = _lib().oracle_fp8_group_params(_p(src_bits), src_bits.shape[1], _p(src_row), _p(group), src_row.size,
                                        int(ngroups), _p(params))
    if rc != 0:
        raise ValueError("oracle_fp8_group_params failed")
    return params[:ngroups]


def quantize_rows_with_params(src_bits, src_row, group, params):
    """(codes uint8 [n, H], scales float32 [n, 2]) of the listed rows."""
    src_bits = _c(src_bits, np.uint16)
    src_row = _c(src_row, np.int64)
    group = _c(group, np.int32)
    params = _c(params, np.float32)
    H = src_bits.shape[1]
    codes = np.empty((src_row.size, H), np.uint8)
    scales = np.empty((src_row.size, 2), np.float32)
    _lib().oracle_quantize_rows_with_params(_p(src_bits), H, _p(src_row), _p(group), src_row.size, _p(params),
                                            _p(codes), _p(scales))
    return codes, scales


def quantize_rows_grouped(src_bits, src_row, group, ngroups):
    """Group parameters over all listed rows, then every row encoded."""
    params = fp8_group_params(src_bits, src_row, group, ngroups)
    return quantize_rows_with_params(src_bits, src_row, group, params)


def row_groups(mode, offsets, rows):
    """(group id per packed row, number of groups) for a quantiser mode:
    per-token = the row itself, per-expert = the row's expert (from the
    layout offsets), global = one group."""
    rows = np.asarray(rows, np.int64)
    offsets = np.asarray(offsets, np.int64)
    if mode == FP8_PER_TOKEN:
        return rows.astype(np.int32), int(rows.max()) + 1 if rows.size else 0
    if mode == FP8_PER_EXPERT:
        E = offsets.size - 1
        return (np.searchsorted(offsets, rows, side="right") - 1).astype(np.int32), E
    if mode == FP8_GLOBAL:
        return np.zeros(rows.size, np.int32), 1
    raise ValueError("unknown FP8 mode")


def combine_fp8_f32order(codes, scales, gates_f32, dst_row, tokens, T, k, shared_bits=None):
    """bf16 bits [n, H] of y from FP8 expert-output rows, pinned fp32 order."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    gates_f32 = _c(gates_f32, np.float32)
    dst_row = _c(dst_row, np.int32)
    tokens = _c(tokens, np.int64)
    H = codes.shape[1]
    sh, Ks = _shared_args(shared_bits, T, H)
    y = np.empty((tokens.size, H), np.uint16)
    _lib().oracle_combine_fp8_f32order_tokens(_p(codes), _p(scales), H, k, _p(gates_f32), _p(dst_row), _p(sh), Ks,
                                              T, _p(tokens), tokens.size, _p(y))
    return y


def combine_fp8_ref64(codes, scales, gates_f32, dst_row, tokens, T, k, shared_bits=None):
    """(fp64 reference [n, H], sum of |terms| [n, H]) of the FP8 combine."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    gates_f32 = _c(gates_f32, np.float32)
    dst_row = _c(dst_row, np.int32)
    tokens = _c(tokens, np.int64)
    H = codes.shape[1]
    sh, Ks = _shared_args(shared_bits, T, H)
    ref = np.empty((tokens.size, H), np.float64)
    mag = np.empty((tokens.size, H), np.float64)
    _lib().oracle_combine_fp8_ref64_tokens(_p(codes), _p(scales), H, k, _p(gates_f32), _p(dst_row), _p(sh), Ks, T,
                                           _p(tokens), tokens.size, _p(ref), _p(mag))
    return ref, mag


def _shared_args(shared_bits, T, H):
    if shared_bits is None:
        return None, 0
    shared_bits = _c(shared_bits, np.uint16)
    assert shared_bits.shape[1:] == (T, H)
    return shared_bits, shared_bits.shape[0]


def combine_f32order(eo_bits, gates_f32, dst_row, tokens, T, k, shared_bits=None):
    """bf16 bits [n, H] of y for the listed tokens, pinned fp32 order."""
    eo_bits = _c(eo_bits, np.uint16)
    gates_f32 = _c(gates_f32, np.float32)
    dst_row = _c(dst_row, np.int32)
    tokens = _c(tokens, np.int64)
    H = eo_bits.shape[1]
    sh, Ks = _shared_args(shared_bits, T, H)
    y = np.empty((tokens.size, H), np.uint16)
    _lib().oracle_combine_f32order_tokens(_p(eo_bits), H, k, _p(gates_f32), _p(dst_row),
                                          _p(sh), Ks, T, _p(tokens), tokens.size, _p(y))
    return y


def combine_ref64(eo_bits, gates_f32, dst_row, tokens, T, k, shared_bits=None):
    """(fp64 reference [n, H], sum of |terms| [n, H]) for the listed tokens."""
    eo_bits = _c(eo_bits, np.uint16)
    gates_f32 = _c(gates_f32, np.float32)
    dst_row = _c(dst_row, np.int32)
    tokens = _c(tokens, np.int64)
    H = eo_bits.shape[1]
    sh, Ks = _shared_args(shared_bits, T, H)
    ref = np.empty((tokens.size, H), np.float64)
    mag = np.empty((tokens.size, H), np.float64)
    _lib().oracle_combine_ref64_tokens(_p(eo_bits), H, k, _p(gates_f32), _p(dst_row),
                                       _p(sh), Ks, T, _p(tokens), tokens.size, _p(ref), _p(mag))
    return ref, mag


def combine_backward(dy_bits, eo_bits, gates_f32, dst_row, tokens, k):
    """(d_eo rows bf16 bits [n*k, H] (row i*k+j for slot j of token i;
    zero for dropped slots), d_gates fp64 [n, k]) for the listed tokens."""
    dy_bits = _c(dy_bits, np.uint16)
    eo_bits = _c(eo_bits, np.uint16)
    gates_f32 = _c(gates_f32, np.float32)
    dst_row = _c(dst_row, np.int32)
    tokens = _c(tokens, np.int64)
    H = dy_bits.shape[1]
    d_eo = np.zeros((tokens.size * k, H), np.uint16)
    d_g = np.empty((tokens.size, k), np.float64)
    _lib().oracle_combine_backward_tokens(_p(dy_bits), _p(eo_bits), H, k, _p(gates_f32), _p(dst_row),
                                          _p(tokens), tokens.size, _p(d_eo), _p(d_g))
    return d_eo, d_g


def dispatch_backward(d_packed_bits, dst_row, tokens, k):
    """(dx bf16 bits [n, H] in the pinned fp32 order, dx fp64 [n, H])."""
    d_packed_bits = _c(d_packed_bits, np.uint16)
    dst_row = _c(dst_row, np.int32)
    tokens = _c(tokens, np.int64)
    H = d_packed_bits.shape[1]
    dx = np.empty((tokens.size, H), np.uint16)
    dx64 = np.empty((tokens.size, H), np.float64)
    _lib().oracle_dispatch_backward_tokens(_p(d_packed_bits), H, k, _p(dst_row), _p(tokens), tokens.size,
                                           _p(dx), _p(dx64))
    return dx, dx64


def gate_backward(logits, topk_idx, d_gates, mode):
    """d_logits fp64 [T, E] for L = sum d_gates * gates(logits)."""
    logits = _c(logits, np.float32)
    topk_idx = _c(topk_idx, np.int32)
    d_gates = _c(d_gates, np.float64)
    T, E = logits.shape
    k = topk_idx.shape[1]
    out = np.empty((T, E), np.float64)
    rc = _lib().oracle_gate_backward(_p(logits), _p(topk_idx), _p(d_gates), T, E, k, mode, _p(out))
    if rc != 0:
        raise ValueError("oracle_gate_backward failed")
    return out


def bf16_bits_from_float(v: np.ndarray) -> np.ndarray:
    f = _lib().oracle_bf16_from_float
    flat = _c(v, np.float32).ravel()
    return np.fromiter((f(float(a)) for a in flat), dtype=np.uint16, count=flat.size).reshape(np.shape(v))
