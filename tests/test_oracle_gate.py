"""Pins of the oracle's gate step (top-k, gate weights, counts, aux, entropy)
against hand-worked values, brute force, closed forms and library routines.
None of these re-types the oracle's own code."""
import math

import numpy as np
import pytest
import torch

from conftest import load_golden

pytestmark = pytest.mark.filterwarnings("ignore")


def _hand_logits():
    g = load_golden("hand_worked_route.json")
    rows = [[(-0.0 if v == "-0.0" else float(v)) for v in r] for r in g["logits"]]
    return g, np.array(rows, np.float32)


def test_hand_worked_topk_counts_aux_entropy(oracle):
    g, logits = _hand_logits()
    idx, gates, counts, aux, ent = oracle.gate(logits, g["k"], oracle.TOPK_SOFTMAX)
    assert idx.tolist() == g["topk_idx"]
    assert counts.tolist() == g["expert_counts"]
    assert aux == g["aux_loss"]
    exact = 0.375 * math.log2(8.0 / 3.0) + 0.5 + 0.375
    assert abs(ent - exact) < g["entropy_eps_tolerance"]
    # closed form of the two-way softmax: logistic of the logit gap
    gap = g["gates_topk_softmax"]["row0_logit_gap"]
    g0 = 1.0 / (1.0 + math.exp(-gap))
    assert abs(gates[0, 0] - g0) < 1e-15 and abs(gates[0, 1] - (1 - g0)) < 1e-15
    assert np.all(gates[1:] == 0.5)


def test_hand_worked_softmax_topk_gates(oracle):
    g, logits = _hand_logits()
    idx = oracle.topk(logits, 2)
    gates = oracle.gates(logits, idx, oracle.SOFTMAX_TOPK)
    S0 = math.exp(-1) + 1 + math.exp(-2) + math.exp(-0.5)
    assert abs(gates[0, 0] - 1 / S0) < 1e-15
    assert abs(gates[0, 1] - math.exp(-0.5) / S0) < 1e-15
    S1 = 2 + 2 * math.exp(-2)
    assert np.allclose(gates[1], [1 / S1, 1 / S1], atol=1e-15, rtol=0)
    assert np.all(gates[3] == 0.25)


def _brute_topk(logits, k):
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (40, 16, 4), (30, 32, 8), (17, 64, 8), (9, 5, 5), (12, 256, 16)])
def test_topk_matches_brute_force_with_ties(oracle, rng, T, E, k):
    # coarse integer-valued logits force many ties
    logits = rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    logits[rng.random((T, E)) < 0.1] = -0.0
    assert np.array_equal(oracle.topk(logits, k), _brute_topk(logits, k))


def test_topk_matches_numpy_lexsort(oracle, rng):
    logits = (rng.standard_normal((500, 64)) * 0.5).round(1).astype(np.float32)
    ref = np.empty((500, 8), np.int32)
    for t in range(500):
        ref[t] = np.lexsort((np.arange(64), -logits[t].astype(np.float64)))[:8]
    assert np.array_equal(oracle.topk(logits, 8), ref)


def test_topk_matches_torch_on_tie_free_inputs(oracle, rng):
    logits = rng.standard_normal((300, 32)).astype(np.float32)
    assert all(len(set(r)) == 32 for r in logits.tolist())
    ref = torch.topk(torch.from_numpy(logits), 8, dim=-1).indices.numpy()
    assert np.array_equal(oracle.topk(logits, 8), ref)


def test_topk_special_cases(oracle):
    eq = np.zeros((3, 8), np.float32)
    assert oracle.topk(eq, 3).tolist() == [[0, 1, 2]] * 3
    z = np.array([[-0.0, 0.0, -0.0, 0.0]], np.float32)
    assert oracle.topk(z, 4).tolist() == [[0, 1, 2, 3]]
    full = np.array([[0.5, -2.0, 3.0, 1.0, -0.25]], np.float32)
    assert oracle.topk(full, 5).tolist() == [[2, 3, 0, 4, 1]]
    with pytest.raises(ValueError):
        oracle.topk(np.array([[0.0, float("nan")]], np.float32), 1)


def test_gates_topk_softmax_closed_form_and_sum(oracle, rng):
    logits = rng.standard_normal((200, 16)).astype(np.float32)
    idx = oracle.topk(logits, 2)
    g = oracle.gates(logits, idx, oracle.TOPK_SOFTMAX)
    l0 = np.take_along_axis(logits, idx, 1).astype(np.float64)
    g0 = 1.0 / (1.0 + np.exp(l0[:, 1] - l0[:, 0]))
    assert np.max(np.abs(g[:, 0] - g0)) < 1e-15
    g8 = oracle.gates(logits, oracle.topk(logits, 8), oracle.TOPK_SOFTMAX)
    assert np.max(np.abs(g8.sum(1) - 1.0)) < 1e-14
    assert np.all(np.diff(g8, axis=1) <= 0)  # descending with the logits


def test_gates_softmax_topk_matches_torch_fp64(oracle, rng):
    logits = (rng.standard_normal((256, 32)) * 3).astype(np.float32)
    idx = oracle.topk(logits, 8)
    g = oracle.gates(logits, idx, oracle.SOFTMAX_TOPK)
    probs = torch.softmax(torch.from_numpy(logits).double(), dim=-1).numpy()
    ref = np.take_along_axis(probs, idx, 1)
    assert np.max(np.abs(g - ref)) < 1e-15
    assert np.all(g.sum(1) < 1.0 + 1e-15)


def test_topk_softmax_equals_softmax_then_renorm(oracle, rng):
    """The two published recipes (top-k then softmax; softmax, top-k, then
    renormalise) give the same gates: identity of the two algorithms."""
    logits = rng.standard_normal((256, 16)).astype(np.float32)
    idx = oracle.topk(logits, 4)
    a = oracle.gates(logits, idx, oracle.TOPK_SOFTMAX)
    p = torch.softmax(torch.from_numpy(logits).double(), dim=-1)
    w, sel = torch.topk(p, 4, dim=-1)
    w = w / w.sum(-1, keepdim=True)
    assert np.array_equal(sel.numpy(), idx)
    assert np.max(np.abs(a - w.numpy())) < 1e-12


def test_counts_match_bincount_and_sum(oracle, rng):
    idx = np.stack([rng.permutation(64)[:8] for _ in range(1000)]).astype(np.int32)
    counts, aux, ent = oracle.stats(idx, 64)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=64))
    assert counts.sum() == idx.size


def test_aux_closed_forms(oracle):
    T, E, k = 64, 8, 2
    # uniform: every expert gets exactly T*k/E assignments -> aux = k^2
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)], np.int32)
    c, aux, ent = oracle.stats(idx, E)
    assert np.all(c == T * k // E)
    assert abs(aux - k * k) < 1e-12
    # the 1e-8 inside the log shifts the entropy by about E * 1e-8 / ln 2
    assert abs(ent - math.log2(E)) < 2 * E * 1e-8 / math.log(2)
    # every token picks the same k experts -> aux = E*k, entropy = log2 k
    same = np.tile(np.array([[3, 5]], np.int32), (T, 1))
    c, aux, ent = oracle.stats(same, E)
    assert abs(aux - E * k) < 1e-12
    assert abs(ent - math.log2(k)) < 1e-7
    # the sync-tax guide's TaxMeter quotes "ideal 4.0" for 16 experts
    idx16 = np.array([[t % 16, (t + 8) % 16] for t in range(128)], np.int32)
    assert abs(oracle.stats(idx16, 16)[2] - 4.0) < 2 * 16 * 1e-8 / math.log(2)


def test_aux_lower_bound_cauchy_schwarz(oracle, rng):
    for _ in range(20):
        E, k = 16, 2
        idx = np.stack([rng.choice(E, k, replace=False, p=rng.dirichlet(np.ones(E)))
                        for _ in range(200)]).astype(np.int32)
        assert oracle.stats(idx, E)[1] >= k * k - 1e-12


def test_empty_batch(oracle):
    c, aux, ent = oracle.stats(np.zeros((0, 2), np.int32), 8)
    assert c.tolist() == [0] * 8 and aux == 0.0 and ent == 0.0
