"""Pins of the oracle's backward functions: finite differences of the
forward oracle, adjoint (dot-product) identities, and exact special cases."""
import numpy as np
import pytest

from test_oracle_combine import _bf16_bits, _f


def _route(oracle, rng, T, E, k, P=4, cap=0, mode=0):
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, g64, *_ = oracle.gate(logits, k, mode)
    L = oracle.layout(idx, E, P, cap, gates_f32=g64.astype(np.float32))
    return logits, idx, L


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_gate_backward_matches_finite_differences(oracle, rng, mode, k):
    T, E = 12, 8
    logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    idx = oracle.topk(logits, k)
    dg = rng.standard_normal((T, k))
    dl = oracle.gate_backward(logits, idx, dg, mode)
    h = 1e-3  # logits are fp32: perturb by an exactly representable step
    for t in range(T):
        for e in range(E):
            lp = logits.copy(); lp[t, e] += np.float32(h)
            lm = logits.copy(); lm[t, e] -= np.float32(h)
            if not (np.array_equal(oracle.topk(lp, k), idx) and np.array_equal(oracle.topk(lm, k), idx)):
                continue  # selection changed: not differentiable there
            step = float(lp[t, e]) - float(lm[t, e])
            fd = (np.sum(dg[t] * oracle.gates(lp, idx, mode)[t]) - np.sum(dg[t] * oracle.gates(lm, idx, mode)[t])) / step
            assert abs(fd - dl[t, e]) < 1e-6, (t, e, fd, dl[t, e])
    if mode == 0:  # only the selected logits receive gradient
        mask = np.zeros((T, E), bool)
        np.put_along_axis(mask, idx, True, 1)
        assert np.all(dl[~mask] == 0.0)
    # softmax gradients sum to zero across the experts of a token
    assert np.max(np.abs(dl.sum(1))) < 1e-12


def test_combine_backward_gate_gradient_is_finite_difference(oracle, rng):
    """d_gates = <dy, expert output row>: the derivative of the fp64 combine
    along each gate."""
    T, H, E, k = 10, 64, 8, 2
    logits, idx, L = _route(oracle, rng, T, E, k)
    eo = _bf16_bits(rng, (L["R"], H))
    dy = _bf16_bits(rng, (T, H))
    toks = np.arange(T)
    d_eo, dg = oracle.combine_backward(dy, eo, L["gates"], L["dst_row"], toks, k)
    dyf = _f(dy).astype(np.float64)
    for t in range(T):
        for j in range(k):
            gp = L["gates"].copy(); gp[t, j] += np.float32(0.25)
            y1, _ = oracle.combine_ref64(eo, gp, L["dst_row"], toks, T, k)
            y0, _ = oracle.combine_ref64(eo, L["gates"], L["dst_row"], toks, T, k)
            fd = np.sum(dyf * (y1 - y0)) / (float(gp[t, j]) - float(L["gates"][t, j]))
            assert abs(fd - dg[t, j]) <= 1e-9 * max(1.0, abs(fd))


def test_combine_backward_adjoint_identity(oracle, rng):
    """<combine(eo), dy> = <eo, d_eo> with d_eo = g * dy (fp64 adjoint),
    the bf16 rounding of d_eo aside."""
    T, H, E, k = 40, 128, 16, 4
    logits, idx, L = _route(oracle, rng, T, E, k, cap=9)
    eo = _bf16_bits(rng, (L["R"], H))
    dy = _bf16_bits(rng, (T, H))
    toks = np.arange(T)
    y64, _ = oracle.combine_ref64(eo, L["gates"], L["dst_row"], toks, T, k)
    d_eo, dg = oracle.combine_backward(dy, eo, L["gates"], L["dst_row"], toks, k)
    lhs = np.sum(y64 * _f(dy))
    rhs = 0.0
    for t in range(T):
        for j in range(k):
            r = L["dst_row"][t * k + j]
            if r < 0:
                assert dg[t, j] == 0.0 and not d_eo[t * k + j].any()
                continue
            rhs += np.dot(_f(eo[r]).astype(np.float64), _f(d_eo[t * k + j]).astype(np.float64))
    assert abs(lhs - rhs) <= 2 ** -8 * np.sum(np.abs(y64 * _f(dy))) + 1e-9
    # and d_eo is exactly the fp32 product rounded once to bf16 for a power-of-two gate
    L2 = dict(L); g2 = np.full_like(L["gates"], 0.5)
    d_eo2, _ = oracle.combine_backward(dy, eo, g2, L["dst_row"], toks, k)
    kept = [(t, j) for t in range(T) for j in range(k) if L["dst_row"][t * k + j] >= 0]
    for t, j in kept[:20]:
        assert np.array_equal(_f(d_eo2[t * k + j]), _f(dy[t]) * np.float32(0.5))


def test_dispatch_backward_adjoint_and_exact_cases(oracle, rng):
    T, H, E, k = 30, 64, 8, 2
    logits, idx, L = _route(oracle, rng, T, E, k)
    x = _bf16_bits(rng, (T, H))
    packed = oracle.dispatch_bf16_rows(x, k, L["src_pos"], np.arange(L["R"]))
    dp = _bf16_bits(rng, (L["R"], H))
    toks = np.arange(T)
    dx, dx64 = oracle.dispatch_backward(dp, L["dst_row"], toks, k)
    lhs = np.sum(_f(packed).astype(np.float64) * _f(dp))
    rhs = np.sum(_f(x).astype(np.float64) * dx64)
    assert abs(lhs - rhs) <= 1e-9 * np.sum(np.abs(_f(packed) * _f(dp)))
    # the gradient of the copies of x, summed back: 2x exactly (k = 2, nothing dropped)
    dx2, _ = oracle.dispatch_backward(packed, L["dst_row"], toks, k)
    assert np.array_equal(_f(dx2), _f(x) * np.float32(2.0))
    # dropped slots contribute nothing
    L3 = oracle.layout(idx, E, 4, 20)
    dx3, dx3_64 = oracle.dispatch_backward(dp[:max(L3["R"], 1)], L3["dst_row"], toks, k)
    for t in range(T):
        want = sum(_f(dp[r]).astype(np.float64) for r in L3["dst_row"][t * k:(t + 1) * k] if r >= 0)
        assert np.allclose(dx3_64[t], want if np.ndim(want) else np.zeros(H), rtol=0, atol=0)
