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
