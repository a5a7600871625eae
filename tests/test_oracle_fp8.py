"""Pins of the oracle's FP8 path: OCP E4M3 encodings, torch's float8_e4m3fn
cast (a library routine), hand-worked per-token rows, and invariants."""
import math

import numpy as np
import pytest
import torch

from conftest import dyadic, load_golden


def _bits(vals):
    """bf16 bit patterns of exactly-representable floats."""
    f = np.asarray(vals, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value is not a bf16"
    return (u >> 16).astype(np.uint16)


def test_ocp_points(oracle):
    g = load_golden("ocp_e4m3_points.json")
    for p in g["points"]:
        assert oracle.e4m3(dyadic(p["v"])) == int(p["code"], 16), p
    special = {"-0.0": -0.0, "inf": math.inf, "-inf": -math.inf}
    for p in g["special"]:
        assert oracle.e4m3(special[p["v"]]) == int(p["code"], 16), p


def test_decode_roundtrip_all_codes(oracle):
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3(oracle.e4m3_decode(c)) == c


def _torch_codes(v):
    t = torch.from_numpy(np.clip(v, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_matches_torch_cast_random(oracle, rng):
    parts = [rng.standard_normal(20000) * s for s in (1e-4, 1e-2, 1.0, 30.0, 300.0)]
    v = np.concatenate(parts + [rng.uniform(-600, 600, 5000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_array(v), _torch_codes(v))


def test_matches_torch_cast_bit_pattern_sweep(oracle):
    # every 4099th float32 bit pattern with |v| <= 2^9, both signs (NaNs excluded)
    u = np.arange(0, 0x44000000, 4099, dtype=np.uint64).astype(np.uint32)
    v = np.concatenate([u, u | 0x80000000]).view(np.float32)
    v = v[np.isfinite(v)]
    assert np.array_equal(oracle.e4m3_array(v), _torch_codes(v))


def test_hand_worked_rows(oracle):
    g = load_golden("fp8_token_rows.json")
    for row in g["rows"]:
        x = _bits([dyadic(p) for p in row["x"]])
        codes, scale, zero = oracle.quantize_row_fp8(x)
        assert [int(c, 16) for c in row["codes"]] == codes.tolist(), row["why"]
        assert scale == dyadic(row["scale"]) and zero == dyadic(row["zero"])


def test_signed_zero_rows(oracle):
    _, s, z = oracle.quantize_row_fp8(_bits([0.0, -0.0, 0.0]))
    assert s == 0.0 and z == 0.0 and not math.copysign(1.0, z) < 0
    _, s, z = oracle.quantize_row_fp8(_bits([-0.0, -0.0]))
    assert s == 0.0 and math.copysign(1.0, z) < 0


def test_row_invariants(oracle, rng):
    for _ in range(50):
        H = 256
        f = (rng.standard_normal(H) * rng.uniform(0.01, 100)).astype(np.float32)
        x = (f.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
        xf = (x.astype(np.uint32) << 16).view(np.float32)
        codes, scale, zero = oracle.quantize_row_fp8(x)
        assert codes[np.argmax(xf)] == 0x7E and codes[np.argmin(xf)] == 0xFE
        # dequantised error: at most half an e4m3 step (relative 2^-4) of v,
        # or half the subnormal step, plus fp32 rounding of the affine map
        v = (xf.astype(np.float64) - zero) / scale
        dq = np.array([oracle.e4m3_decode(c) for c in codes])
        step = np.where(np.abs(v) < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 2 ** -6))) - 3))
        assert np.all(np.abs(dq - v) <= 0.5 * step * (1 + 1e-5) + 1e-4)
