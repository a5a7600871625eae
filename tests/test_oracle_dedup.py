"""Pins of the per-partition de-duplication: a hand-worked fixture, the
invariants that tie it to the layout it came from, and the whole
de-duplicated path (send once per partition, expand, partial combine,
return, add) equal to the plain combine where every sum is exact."""
import numpy as np
import pytest

from conftest import load_golden
from test_oracle_combine import _bf16_bits, _f


def test_hand_worked(oracle):
    d = load_golden("dedup_layout.json")
    L = oracle.layout(np.array(d["topk_idx"], np.int32), d["E"], d["P"], 0)
    assert list(L["dst_row"]) == d["dst_row"] and list(L["offsets"]) == d["offsets"]
    D = oracle.dedup_layout(L["dst_row"], L["offsets"], np.array(d["gates"], np.float32), d["T"], d["E"], d["k"],
                            d["P"])
    assert list(D["send_offsets"]) == d["send_offsets"]
    assert D["send_row"].tolist() == d["send_row"]
    assert list(D["send_token"]) == d["send_token"]
    assert D["slot_local"].tolist() == d["slot_local"]
    assert D["slot_gate"].tolist() == d["slot_gate"]


def _final_expert(L, E):
    fe = np.full(L["dst_row"].size, -1)
    ok = L["dst_row"] >= 0
    fe[ok] = np.searchsorted(L["offsets"], L["dst_row"][ok], side="right") - 1
    return fe


@pytest.mark.parametrize("T,E,k,P,cap,reassign", [(80, 16, 4, 4, 0, False), (120, 16, 8, 4, 60, False),
                                                   (150, 32, 6, 8, 25, True), (60, 8, 1, 2, 0, False)])
def test_invariants(oracle, rng, T, E, k, P, cap, reassign):
    logits = rng.standard_normal((T, E)) + 2.0 * np.log(1.0 / (1.0 + rng.permutation(E)))
    idx = np.argsort(-logits, 1, kind="stable")[:, :k].astype(np.int32)
    g = rng.random((T, k)).astype(np.float32)
    L = oracle.layout_reassign(idx, E, P, cap, gates_f32=g) if reassign else oracle.layout(idx, E, P, cap, gates_f32=g)
    D = oracle.dedup_layout(L["dst_row"], L["offsets"], L["gates"], T, E, k, P)
    per = E // P
    fe = _final_expert(L, E).reshape(T, k)
    assert list(np.diff(D["send_offsets"])) == list(L["part_tokens"])
    seen = 0
    for t in range(T):
        for p in range(P):
            slots = [j for j in range(k) if fe[t, j] >= 0 and fe[t, j] // per == p]
            s = D["send_row"][t, p]
            if not slots:
                assert s == -1
                continue
            assert D["send_offsets"][p] <= s < D["send_offsets"][p + 1] and D["send_token"][s] == t
            assert list(D["slot_local"][s][:len(slots)]) == [fe[t, j] - p * per for j in slots]
            assert list(D["slot_gate"][s][:len(slots)]) == [L["gates"][t, j] for j in slots]
            assert np.all(D["slot_local"][s][len(slots):] == -1) and np.all(D["slot_gate"][s][len(slots):] == 0)
            seen += len(slots)
    assert seen == L["R"]
    for p in range(P):  # tokens ascending within a partition
        toks = D["send_token"][D["send_offsets"][p]:D["send_offsets"][p + 1]]
        assert np.all(np.diff(toks) > 0)


def test_deduplicated_path_equals_plain_combine_when_exact(oracle, rng):
    """Identity experts, gates in multiples of 1/8, x in multiples of 1/16
    with small magnitude: every partial and total sum is exact in fp32 and
    bf16, so sending once per partition (expand on the receiver, combine
    there, add the partials at the source) must give the plain combine."""
    T, E, k, P, H = 64, 16, 4, 4, 32
    logits = rng.standard_normal((T, E))
    idx = np.argsort(-logits, 1, kind="stable")[:, :k].astype(np.int32)
    g = (rng.integers(1, 8, (T, k)) / 8.0).astype(np.float32)
    L = oracle.layout(idx, E, P, 0, gates_f32=g)
    xf = (rng.integers(-16, 17, (T, H)) / 16.0).astype(np.float32)
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)
    packed = oracle.dispatch_bf16_rows(x, k, L["src_pos"], np.arange(L["R"]))
    y_plain = oracle.combine_f32order(packed, L["gates"], L["dst_row"], np.arange(T), T, k)
    D = oracle.dedup_layout(L["dst_row"], L["offsets"], L["gates"], T, E, k, P)
    per = E // P
    partials = []
    for p in range(P):
        s0, s1 = D["send_offsets"][p], D["send_offsets"][p + 1]
        recv = x[D["send_token"][s0:s1]]
        Lp = oracle.layout(D["slot_local"][s0:s1], per, 1, 0)
        local = oracle.dispatch_bf16_rows(recv, k, Lp["src_pos"], np.arange(Lp["R"]))
        part = oracle.combine_f32order(local, D["slot_gate"][s0:s1], Lp["dst_row"], np.arange(s1 - s0), s1 - s0, k)
        partials.append(part)
    partials = np.concatenate(partials)
    y_dedup = oracle.combine_f32order(partials, np.ones((T, P), np.float32), D["send_row"].ravel(), np.arange(T), T, P)
    assert np.array_equal(y_dedup, y_plain)
    # and the receive-side layouts see every kept slot once
    assert sum(oracle.layout(D["slot_local"][D["send_offsets"][p]:D["send_offsets"][p + 1]], per, 1, 0)["R"]
               for p in range(P)) == L["R"]
