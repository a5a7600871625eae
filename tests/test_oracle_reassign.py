"""Pins of the re-assigning layout: hand-worked fixtures, the closed form
of the water filling (an independent characterisation of pass 2), its
agreement with the dropping layout on the kept assignments, and the
invariants of a layout."""
import numpy as np
import pytest

from conftest import load_golden


@pytest.mark.parametrize("case", range(2))
def test_hand_worked(oracle, case):
    c = load_golden("reassign_layout.json")["cases"][case]
    idx = np.array(c["topk_idx"], np.int32)
    L = oracle.layout_reassign(idx, c["E"], c["P"], c["capacity"])
    for key in ("counts", "offsets", "dst_row", "src_pos", "capacity_mask", "final_expert", "part_rows",
                "part_offsets", "part_tokens"):
        assert list(L[key]) == c[key], key
    assert L["dropped"] == c["dropped"]


def water_fill_loads(L, O, C):
    """Final loads when O assignments go one at a time to the lowest-loaded
    expert below C (ties to the lower id), in closed form: the slots (level,
    expert) with level in [L_e, C) are taken in (level, expert) order, so
    the loads are the first O of those slots counted per expert."""
    slots = sorted((lev, e) for e, l0 in enumerate(L) for lev in range(l0, C))
    out = list(L)
    for lev, e in slots[:O]:
        out[e] += 1
    return out


def _skewed_ids(rng, T, E, k, hot=3.0):
    logits = rng.standard_normal((T, E)) + hot * np.log(1.0 / (1.0 + rng.permutation(E)))
    return np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)


@pytest.mark.parametrize("T,E,k,C", [(60, 8, 2, 10), (200, 16, 4, 40), (97, 5, 3, 30), (50, 4, 2, 20),
                                     (40, 8, 8, 30)])
def test_closed_form_and_invariants(oracle, rng, T, E, k, C):
    idx = _skewed_ids(rng, T, E, k)
    P = 1 if E % 2 else 2
    g = rng.random((T, k)).astype(np.float32)
    L = oracle.layout_reassign(idx, E, P, C, gates_f32=g)
    D = oracle.layout(idx, E, P, C)
    A = T * k
    raw = np.bincount(idx.ravel(), minlength=E)
    kept = np.minimum(raw, C)
    O = int(np.sum(raw - kept))
    assert list(L["counts"]) == water_fill_loads(list(kept), O, C)
    assert L["R"] == min(A, E * C) and L["dropped"] == A - L["R"]
    assert np.all(L["counts"] <= C)
    # pass 1 is the dropping layout: same kept set, same order at the head of each expert
    direct = L["capacity_mask"] == 1
    assert np.array_equal(direct, D["capacity_mask"] == 1)
    fe = L["final_expert"]
    assert np.array_equal(fe[direct], idx.ravel()[direct])
    rank_l = L["dst_row"][direct] - L["offsets"][fe[direct]]
    rank_d = D["dst_row"][direct] - D["offsets"][idx.ravel()[direct]]
    assert np.array_equal(rank_l, rank_d)
    # pass 2: levels never go down in flat order; within a level, experts by id
    re = np.flatnonzero(L["capacity_mask"] == 2)
    lev = L["dst_row"][re] - L["offsets"][fe[re]]
    key = lev.astype(np.int64) * E + fe[re]
    assert np.all(np.diff(key) > 0)
    assert np.all(lev >= kept[fe[re]])
    # a bijection between kept assignments and rows
    ok = fe >= 0
    assert np.array_equal(np.sort(L["dst_row"][ok]), np.arange(L["R"]))
    assert np.array_equal(L["src_pos"][L["dst_row"][ok]], np.flatnonzero(ok))
    assert np.all(L["dst_row"][~ok] == -1) and np.all(L["capacity_mask"][~ok] == 0)
    # gates: only dropped slots are zeroed
    gz = L["gates"].ravel()
    assert np.array_equal(gz[ok], g.ravel()[ok]) and np.all(gz[~ok] == 0)
    # partitions from the final experts
    per = E // P
    want = [sum(1 for t in range(T) if any(fe[t * k + j] >= 0 and fe[t * k + j] // per == p for j in range(k)))
            for p in range(P)]
    assert list(L["part_tokens"]) == want
    assert list(L["part_rows"]) == [int(L["counts"][p * per:(p + 1) * per].sum()) for p in range(P)]


def test_no_overflow_equals_dropping_layout(oracle, rng):
    idx = _skewed_ids(rng, 50, 8, 2, hot=0.0)
    L = oracle.layout_reassign(idx, 8, 4, 1000)
    D = oracle.layout(idx, 8, 4, 1000)
    for key in ("counts", "offsets", "dst_row", "src_pos", "part_rows", "part_offsets", "part_tokens"):
        assert np.array_equal(L[key], D[key]), key
