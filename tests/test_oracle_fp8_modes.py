"""Pins of the grouped FP8 quantiser (per-token / per-expert / global) and
of the FP8 combine, against the pinned per-token quantiser, the definition
of a group (the concatenation of its rows), a hand-worked fixture and the
fp64 error bound."""
import numpy as np
import pytest

from conftest import load_golden
from test_oracle_combine import _bf16_bits, _f


def _bits_of(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_per_token_groups_equal_the_per_token_quantiser(oracle, rng):
    x = _bf16_bits(rng, (12, 48))
    x[3] = x[3, 0]            # a constant row
    x[5, :] = 0x8000          # a -0 row
    rows = np.arange(12)
    codes, scales = oracle.quantize_rows_grouped(x, rows, rows.astype(np.int32), 12)
    for i in range(12):
        c, s, z = oracle.quantize_row_fp8(x[i])
        assert np.array_equal(codes[i], c)
        assert scales[i, 0] == np.float32(s) and scales[i, 1] == np.float32(z)


@pytest.mark.parametrize("ngroups", [1, 3])
def test_a_group_quantises_like_the_concatenation_of_its_rows(oracle, rng, ngroups):
    x = (_bf16_bits(rng, (30, 16)))
    x[7] = _bits_of(np.full(16, 9.5))  # an outlier row widens its group's range
    src_row = rng.permutation(30)[:20].astype(np.int64)
    group = (np.arange(20) % ngroups).astype(np.int32)
    codes, scales = oracle.quantize_rows_grouped(x, src_row, group, ngroups)
    for g in range(ngroups):
        sel = np.flatnonzero(group == g)
        cat = x[src_row[sel]].reshape(-1)
        c, s, z = oracle.quantize_row_fp8(cat)
        assert np.array_equal(codes[sel].reshape(-1), c)
        assert np.all(scales[sel, 0] == np.float32(s)) and np.all(scales[sel, 1] == np.float32(z))


def test_group_params_of_empty_and_constant_groups(oracle):
    x = _bits_of(np.array([[2.0, 2.0], [2.0, 2.0], [-1.0, 3.0]]))
    p = oracle.fp8_group_params(x, np.array([0, 1, 2]), np.array([0, 0, 2], np.int32), 3)
    assert p[0, 0] == 0.0 and p[0, 1] == 2.0      # constant group: scale 0
    assert p[1, 0] == 0.0 and p[1, 1] == 0.0      # no rows
    assert p[2, 1] == 1.0 and p[2, 0] == np.float32(4.0) / np.float32(896.0)
    codes, sc = oracle.quantize_rows_with_params(x, np.array([0, 2]), np.array([0, 2], np.int32), p)
    assert not codes[0].any()
    assert codes[1, 0] == 0xFE and codes[1, 1] == 0x7E   # min -> -448, max -> +448


def test_row_groups_follow_the_layout(oracle, rng):
    offsets = np.array([0, 3, 3, 7, 10])
    rows = np.arange(10)
    g, n = oracle.row_groups(oracle.FP8_PER_EXPERT, offsets, rows)
    assert n == 4 and list(g) == [0, 0, 0, 2, 2, 2, 2, 3, 3, 3]
    g, n = oracle.row_groups(oracle.FP8_GLOBAL, offsets, rows)
    assert n == 1 and not g.any()
    g, n = oracle.row_groups(oracle.FP8_PER_TOKEN, offsets, rows)
    assert list(g) == list(range(10))


def test_fp8_combine_hand_worked(oracle):
    d = load_golden("fp8_combine_rows.json")
    codes = np.array(d["codes"], np.uint8)
    scales = np.array(d["scales"], np.float32)
    gates = np.array(d["gates"], np.float32)
    dst = np.array(d["dst_row"], np.int32)
    shared = _bits_of(np.array(d["shared"], np.float32))
    toks = np.arange(2)
    # the dequantised values first: zero + scale * value
    deq = np.array([[scales[r, 1] + scales[r, 0] * oracle.e4m3_decode(c) for c in codes[r]] for r in range(3)])
    assert np.array_equal(deq, np.array(d["dequantised"]))
    y = oracle.combine_fp8_f32order(codes, scales, gates, dst, toks, 2, d["k"], shared)
    assert np.array_equal(y, np.array(d["y_bf16_bits"], np.uint16))
    assert np.array_equal(_f(y), np.array(d["y"], np.float32))
    ref, _ = oracle.combine_fp8_ref64(codes, scales, gates, dst, toks, 2, d["k"], shared)
    assert np.array_equal(ref, np.array(d["y"]))


def _ulp_bf16(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return 2.0 ** (np.maximum(e, -126) - 7)


def test_fp8_combine_within_the_fp64_bound_and_close_to_bf16(oracle, rng):
    T, H, E, k, Ks = 40, 64, 8, 2, 1
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, g64, *_ = oracle.gate(logits, k, 0)
    L = oracle.layout(idx, E, 4, 9, gates_f32=g64.astype(np.float32))
    eo = _bf16_bits(rng, (L["R"], H))
    rows = np.arange(L["R"])
    codes, scales = oracle.quantize_rows_grouped(eo, rows, rows.astype(np.int32), L["R"])
    shared = _bf16_bits(rng, (Ks, T, H))
    toks = np.arange(T)
    y = oracle.combine_fp8_f32order(codes, scales, L["gates"], L["dst_row"], toks, T, k, shared)
    ref, mag = oracle.combine_fp8_ref64(codes, scales, L["gates"], L["dst_row"], toks, T, k, shared)
    err = np.abs(_f(y).astype(np.float64) - ref)
    assert np.all(err <= _ulp_bf16(ref) + (k + Ks + 1) * 2.0 ** -24 * mag)
    # against the bf16 combine of the unquantised rows: the quantisation error
    # of e4m3 (3 mantissa bits: |q - e4m3(q)| <= 2^-4 |q|, or 2^-10 below 2^-6)
    # scaled back by each row's scale, plus the rounding terms
    y16, _ = oracle.combine_ref64(eo, L["gates"], L["dst_row"], toks, T, k, shared)
    dq = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            r = L["dst_row"][t * k + j]
            if r < 0:
                continue
            q = np.abs((_f(eo[r]).astype(np.float64) - scales[r, 1]) / max(scales[r, 0], 1e-30))
            dq[t] += abs(L["gates"][t, j]) * scales[r, 0] * np.maximum(q * 2.0 ** -4, 2.0 ** -10) * 1.001
    assert np.all(np.abs(ref - y16) <= dq + 1e-6)
