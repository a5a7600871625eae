"""Pins of the oracle's dispatch layout: the hand-worked fixture, a library
stable argsort, and the invariants the layout must satisfy (bijection,
monotone offsets, token order within an expert, capacity, partitions)."""
import numpy as np
import pytest

from conftest import load_golden


def _hand_idx():
    g = load_golden("hand_worked_route.json")
    return g, np.array(g["topk_idx"], np.int32)


@pytest.mark.parametrize("key,cap", [("layout_no_capacity", 0), ("layout_capacity_3", 3)])
def test_hand_worked_layout(oracle, key, cap):
    g, idx = _hand_idx()
    want = g[key]
    gates = np.full((4, 2), 0.5, np.float32)
    L = oracle.layout(idx, g["E"], g["P"], cap, gates_f32=gates)
    for name in ["counts", "offsets", "dst_row", "src_pos", "capacity_mask", "part_rows",
                 "part_offsets", "part_tokens"]:
        assert L[name].tolist() == want[name], name
    assert L["dropped"] == want["dropped"]
    zeroed = sorted(np.flatnonzero(L["gates"].ravel() == 0).tolist())
    assert zeroed == want.get("gates_zeroed", [])


def _check_invariants(idx, E, P, cap, L):
    T, k = idx.shape
    A = T * k
    flat = idx.ravel()
    counts = np.bincount(flat, minlength=E)
    kc = counts if cap <= 0 else np.minimum(counts, cap)
    assert np.array_equal(L["counts"], kc)
    assert L["offsets"][0] == 0 and np.all(np.diff(L["offsets"]) == kc)
    R = int(L["offsets"][E])
    assert L["R"] == R and L["dropped"] == A - R
    kept = L["dst_row"] >= 0
    assert np.array_equal(kept.astype(np.uint8), L["capacity_mask"])
    # bijection kept assignments <-> [0, R)
    rows = L["dst_row"][kept]
    assert np.array_equal(np.sort(rows), np.arange(R))
    assert np.array_equal(L["src_pos"][L["dst_row"][kept]], np.flatnonzero(kept))
    # packed rows are expert-contiguous, in token order inside an expert
    e_of_row = flat[L["src_pos"]]
    assert np.all(np.diff(e_of_row) >= 0)
    for e in range(E):
        seg = L["src_pos"][L["offsets"][e]:L["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)
    # drops are exactly the assignments whose rank within the expert is >= cap
    order = np.argsort(flat, kind="stable")
    rank = np.empty(A, np.int64)
    start = np.concatenate([[0], np.cumsum(counts)])
    rank[order] = np.arange(A) - start[flat[order]]
    want_kept = np.ones(A, bool) if cap <= 0 else rank < cap
    assert np.array_equal(kept, want_kept)
    # partitions
    per = E // P
    assert np.array_equal(L["part_offsets"], L["offsets"][::per])
    assert np.array_equal(L["part_rows"], np.add.reduceat(kc, np.arange(0, E, per)))
    assert L["part_rows"].sum() == R
    want_tok = [len({t for t in range(T) if any(kept[t * k + j] and flat[t * k + j] // per == p
                                                 for j in range(k))}) for p in range(P)]
    assert L["part_tokens"].tolist() == want_tok


def _random_idx(rng, T, E, k, skew=0.0):
    w = np.exp(-skew * np.arange(E)) if skew else np.ones(E)
    w = w / w.sum()
    return np.stack([rng.choice(E, k, replace=False, p=w) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,P,cap,skew", [
    (256, 8, 2, 4, 0, 0.0),
    (300, 16, 2, 4, 0, 0.0),
    (200, 32, 8, 8, 0, 0.0),
    (500, 64, 2, 8, 0, 0.3),
    (400, 64, 8, 8, 63, 0.2),     # ceil(1.25*T*k/E) = 63
    (100, 8, 2, 2, 1, 0.0),       # capacity 1
    (77, 16, 4, 16, 5, 1.0),      # heavy skew, one expert per partition
])
def test_layout_invariants(oracle, rng, T, E, k, P, cap, skew):
    idx = _random_idx(rng, T, E, k, skew)
    L = oracle.layout(idx, E, P, cap)
    _check_invariants(idx, E, P, cap, L)


def test_layout_permutation_is_stable_argsort(oracle, rng):
    idx = _random_idx(rng, 1000, 16, 2, 0.1)
    L = oracle.layout(idx, 16, 4, 0)
    assert np.array_equal(L["src_pos"], np.argsort(idx.ravel(), kind="stable"))


def test_layout_all_tokens_one_expert_and_exact_capacity(oracle):
    T, E, k = 50, 8, 2
    idx = np.tile(np.array([[6, 2]], np.int32), (T, 1))
    L = oracle.layout(idx, E, 4, T)          # capacity exactly hit: nothing dropped
    assert L["dropped"] == 0 and L["counts"].tolist() == [0, 0, T, 0, 0, 0, T, 0]
    _check_invariants(idx, E, 4, T, L)
    L = oracle.layout(idx, E, 4, T - 1)      # one over: the last token loses both slots
    assert L["dropped"] == 2 and L["dst_row"][-2:].tolist() == [-1, -1]
    _check_invariants(idx, E, 4, T - 1, L)


def test_layout_k_equals_E(oracle, rng):
    idx = np.stack([rng.permutation(8) for _ in range(33)]).astype(np.int32)
    L = oracle.layout(idx, 8, 8, 0)
    _check_invariants(idx, 8, 8, 0, L)
    assert L["part_tokens"].tolist() == [33] * 8


def test_layout_empty(oracle):
    L = oracle.layout(np.zeros((0, 2), np.int32), 8, 4, 0)
    assert L["R"] == 0 and L["offsets"].tolist() == [0] * 9 and L["part_tokens"].tolist() == [0] * 4


def test_layout_rejects_bad_ids(oracle):
    with pytest.raises(ValueError):
        oracle.layout(np.array([[0, 9]], np.int32), 8, 4, 0)
