"""Pins of the oracle's dispatch (bf16) and combine: the identity-expert
round trip, the hand-worked fixture, and the fp64 error bound."""
import numpy as np
import pytest

from conftest import load_golden


def _bf16_bits(rng, shape, scale=1.0):
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    u = f.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _pipeline(oracle, logits, x, k, P, cap, mode):
    E = logits.shape[1]
    T = x.shape[0]
    idx, g64, counts, aux, ent = oracle.gate(logits, k, mode)
    L = oracle.layout(idx, E, P, cap, gates_f32=g64.astype(np.float32))
    packed = oracle.dispatch_bf16_rows(x, k, L["src_pos"], np.arange(L["R"]))
    return idx, L, packed


@pytest.mark.parametrize("T,H,E,k,P", [(256, 512, 8, 2, 4), (64, 256, 16, 4, 4), (40, 128, 32, 8, 8)])
def test_identity_experts_round_trip(oracle, rng, T, H, E, k, P):
    """combine(dispatch(x)) == x bit-exactly when each expert is the
    identity and the gates sum to one (top-k-then-softmax, no drops)."""
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = _bf16_bits(rng, (T, H))
    idx, L, packed = _pipeline(oracle, logits, x, k, P, 0, oracle.TOPK_SOFTMAX)
    y = oracle.combine_f32order(packed, L["gates"], L["dst_row"], np.arange(T), T, k)
    assert np.array_equal(y, x)


def test_hand_worked_combine(oracle, rng):
    g = load_golden("hand_worked_route.json")
    idx = np.array(g["topk_idx"], np.int32)
    x = _bf16_bits(rng, (4, 64))
    logits = np.array([[0.0, 1.0, -1.0, 0.5], [2, 2, 0, 0], [-0.0, 0, -3, -3], [0, 0, 0, 0]], np.float32)
    gates = oracle.gates(logits, idx, oracle.TOPK_SOFTMAX).astype(np.float32)
    for cap in (0, 3):
        L = oracle.layout(idx, 4, 2, cap, gates_f32=gates)
        packed = oracle.dispatch_bf16_rows(x, 2, L["src_pos"], np.arange(L["R"]))
        y = oracle.combine_f32order(packed, L["gates"], L["dst_row"], np.arange(4), 4, 2)
        if cap == 0:
            assert np.array_equal(y, x)
        else:
            assert np.array_equal(y[:3], x[:3])
            assert np.array_equal(_f(y[3]), _f(x[3]) * np.float32(0.5))


def test_dispatch_rows_are_token_copies(oracle, rng):
    T, H, E, k = 100, 64, 8, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = _bf16_bits(rng, (T, H))
    idx, L, packed = _pipeline(oracle, logits, x, k, 4, 0, oracle.TOPK_SOFTMAX)
    for r in range(L["R"]):
        assert np.array_equal(packed[r], x[L["src_pos"][r] // k])


def _ulp_bf16(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return 2.0 ** (np.maximum(e, -126) - 7)


@pytest.mark.parametrize("k,Ks,cap", [(2, 0, 0), (8, 2, 0), (8, 0, 40)])
def test_f32order_within_bound_of_fp64_reference(oracle, rng, k, Ks, cap):
    T, H, E = 80, 256, 32
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, g64, *_ = oracle.gate(logits, k, oracle.SOFTMAX_TOPK)
    L = oracle.layout(idx, E, 8, cap, gates_f32=g64.astype(np.float32))
    eo = _bf16_bits(rng, (max(L["R"], 1), H))
    shared = _bf16_bits(rng, (Ks, T, H)) if Ks else None
    toks = np.arange(T)
    y = oracle.combine_f32order(eo, L["gates"], L["dst_row"], toks, T, k, shared)
    ref, mag = oracle.combine_ref64(eo, L["gates"], L["dst_row"], toks, T, k, shared)
    n = k + Ks
    err = np.abs(_f(y).astype(np.float64) - ref)
    bound = _ulp_bf16(ref) + n * 2.0 ** -24 * mag
    assert np.all(err <= bound)
    # most outputs are within one bf16 ulp of the fp64 reference
    assert np.mean(err <= _ulp_bf16(ref)) > 0.999


def test_dropped_slots_do_not_contribute(oracle, rng):
    T, H, k = 6, 32, 2
    eo = _bf16_bits(rng, (12, H))
    gates = np.full((T, k), 0.5, np.float32)
    dst = np.arange(T * k, dtype=np.int32)
    dst[1] = -1
    y = oracle.combine_f32order(eo, gates, dst, np.arange(T), T, k)
    assert np.array_equal(_f(y[0]), _f(eo[0]) * np.float32(0.5))


def _f32_to_bf16_exact(v):
    """bf16 bits of values that are exact in bf16 (asserted)."""
    u = np.asarray(v, np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "fixture value not exact in bf16"
    return (u >> 16).astype(np.uint16)


@pytest.mark.parametrize("case", [0, 1])
def test_hand_worked_shared_expert_combine(oracle, case):
    """Shared experts (K_s = 2 and 3) added with weight 1 after the routed
    terms, against hand-worked values: both the pinned fp32 order and the
    fp64 reference must give the fixture's y exactly (every term and partial
    sum is dyadic).  The shared rows differ per (s, t), so a transposed
    [t, s] index or a dropped last shared expert fails here."""
    g = load_golden("shared_expert_combine.json")
    c = g["cases"][case]
    T, Ks, k, H = c["T"], c["Ks"], g["k"], g["H"]
    eo = _f32_to_bf16_exact(g["expert_rows"])
    gates = np.array(c["gates"], np.float32)
    dst = np.array(c["dst_row"], np.int32)
    shared = _f32_to_bf16_exact(c["shared"])
    assert shared.shape == (Ks, T, H)
    toks = np.arange(T)
    want = np.array(c["y"], np.float32)
    y = oracle.combine_f32order(eo, gates, dst, toks, T, k, shared)
    assert np.array_equal(_f(y), want)
    ref, mag = oracle.combine_ref64(eo, gates, dst, toks, T, k, shared)
    assert np.array_equal(ref, want.astype(np.float64))
    # without the shared experts only the routed terms remain
    y0 = oracle.combine_f32order(eo, gates, dst, toks, T, k, None)
    assert np.array_equal(_f(y0), np.array(c["routed_only"], np.float32))
    if "abs_terms_token1" in c:
        assert np.array_equal(mag[1], np.array(c["abs_terms_token1"], np.float64))
    # a subset of tokens reads the same shared rows (token index, not position in the list)
    y1 = oracle.combine_f32order(eo, gates, dst, np.array([T - 1]), T, k, shared)
    assert np.array_equal(_f(y1[0]), want[T - 1])


@pytest.mark.parametrize("case", [0, 1])
def test_hand_worked_shared_expert_combine_fp8(oracle, case):
    """The FP8 combine on the same rows given as e4m3 codes with (scale,
    zero) = (1, 0): the same hand-worked y, shared experts included."""
    g = load_golden("shared_expert_combine.json")
    c = g["cases"][case]
    T, Ks, k = c["T"], c["Ks"], g["k"]
    codes = np.array(g["expert_rows_e4m3"], np.uint8)
    assert np.array_equal(np.array([[oracle.e4m3_decode(int(v)) for v in r] for r in codes]),
                          np.array(g["expert_rows"], np.float64))
    scales = np.tile(np.array([1.0, 0.0], np.float32), (codes.shape[0], 1))
    gates = np.array(c["gates"], np.float32)
    dst = np.array(c["dst_row"], np.int32)
    shared = _f32_to_bf16_exact(c["shared"])
    toks = np.arange(T)
    want = np.array(c["y"], np.float32)
    y = oracle.combine_fp8_f32order(codes, scales, gates, dst, toks, T, k, shared)
    assert np.array_equal(_f(y), want)
    ref, _ = oracle.combine_fp8_ref64(codes, scales, gates, dst, toks, T, k, shared)
    assert np.array_equal(ref, want.astype(np.float64))
