"""GPU parity of the backward calls against the oracle, on the forward
layout of the same seeded workloads.

Bit-exact: d_expert_out rows (one fp32 product, one bf16 rounding) and dx
(fp32 sum of the kept copies' gradients in slot order).  d_gates within the
fp32 summation bound the header states, (H/256 + 14) * 2^-24 * sum|dy*eo|,
and exactly 0 for dropped slots.  d_logits within a bound derived from the
fp32 softmax recomputation: 2 * (max|l - m| + E + k + 8) * 2^-24 times the
magnitude of the terms of each element.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import workloads
from gpu_util import bits, check_gate, check_layout, f_of_bits, run_gpu, sample_rows

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()
    torch.cuda.init()


def _gather(t, rows):
    if rows.size == 0:
        return np.zeros((1, t.shape[-1]), np.uint16)
    return bits(t.index_select(0, torch.from_numpy(rows.astype(np.int64)).to(t.device)))


def _check_backward(w, token_sample=None, seed=11):
    """Forward on the GPU (gate compared, oracle gates swapped in, layout
    compared), then the backward calls on seeded gradients; the oracle gets
    its own layout and gates and the same seeded tensors."""
    rng = np.random.default_rng(seed)
    inp = workloads.make_inputs(w, "cuda")
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp)
    assert status == 0
    check_gate(w, plan, gates_pre, og)
    L = check_layout(w, plan, og)
    dy = workloads.make_dy(w, "cuda")
    dp = workloads.make_d_packed(w, max(R, 1), "cuda")
    dg_in = workloads.make_d_gates(w, "cuda")
    plan.combine_backward(dy, eo)
    plan.gate_backward(inp["logits"], dg_in)
    plan.dispatch_backward(dp)
    assert plan.status() == 0, "device status after the backward"
    T, k, H, E = w.T, w.k, w.H, w.E
    if T == 0:
        return plan
    toks = np.arange(T, dtype=np.int64) if token_sample is None else sample_rows(T, rng, token_sample)
    n = toks.size
    dst = L["dst_row"].reshape(T, k)[toks]
    need = np.unique(dst[dst >= 0])
    remap = np.where(dst >= 0, np.searchsorted(need, np.maximum(dst, 0)), -1).astype(np.int32).ravel()
    dy_c = _gather(dy, toks)
    g_c = L["gates"][toks]
    eo_rows = _gather(eo, need) if not w.identity_experts else \
        (oracle.dispatch_bf16_rows(bits(inp["x"]), k, L["src_pos"], need) if need.size else _gather(eo, need))

    # combine backward
    d_eo_ref, dg_ref = oracle.combine_backward(dy_c, eo_rows, g_c, remap, np.arange(n), k)
    got_rows = _gather(plan.d_expert_out, need)
    kept = dst.ravel() >= 0
    assert np.array_equal(got_rows[remap[kept]], d_eo_ref[kept]), "d_expert_out differs from the oracle"
    dg = plan.d_gates.cpu().numpy()[:T][toks]
    assert np.all(dg.ravel()[~kept] == 0.0), "dropped slots must get a zero gate gradient"
    eo_c = f_of_bits(eo_rows).astype(np.float64)
    dyf = f_of_bits(dy_c).astype(np.float64)
    mag = np.zeros(n * k)
    for i in np.flatnonzero(kept):
        mag[i] = np.sum(np.abs(dyf[i // k] * eo_c[remap[i]]))
    bound = (H / 256 + 14) * 2.0 ** -24 * mag + 1e-30
    err = np.abs(dg.ravel().astype(np.float64) - dg_ref.ravel())
    assert np.all(err <= bound), f"d_gates outside the fp32 bound: worst {np.max(err / bound)} x bound"

    # dispatch backward
    dx_ref, dx64 = oracle.dispatch_backward(_gather(dp, need), remap, np.arange(n), k)
    dx = _gather(plan.dx, toks)
    assert np.array_equal(dx, dx_ref), f"dx differs from the oracle in {np.sum(dx != dx_ref)} values"
    none_kept = ~kept.reshape(n, k).any(1)
    assert not np.any(dx[none_kept]), "a token with no kept slot has dx = 0"

    # gate backward on the seeded gate gradients
    logits = inp["logits"].cpu().numpy()[toks]
    idx = og[0][toks]
    dgs = dg_in.cpu().numpy()[toks].astype(np.float64)
    dl_ref = oracle.gate_backward(logits, idx, dgs, w.mode)
    dl = plan.d_logits.cpu().numpy()[:T][toks].astype(np.float64)
    l64 = logits.astype(np.float64)
    sel = np.zeros((n, E), bool)
    np.put_along_axis(sel, idx, True, 1)
    dsel = np.zeros((n, E))
    np.put_along_axis(dsel, idx, np.abs(dgs), 1)
    if w.mode == workloads.TOPK_SOFTMAX:
        lm = np.where(sel, l64, -np.inf)
        m = lm.max(1, keepdims=True)
        p = np.where(sel, np.exp(lm - m), 0.0)
        rng_l = np.where(sel, np.abs(l64 - m), 0.0).max(1, keepdims=True)
    else:
        m = l64.max(1, keepdims=True)
        p = np.exp(l64 - m)
        rng_l = np.abs(l64 - m).max(1, keepdims=True)
    p /= p.sum(1, keepdims=True)
    g_sel = np.take_along_axis(p, idx, 1)
    S1 = np.sum(g_sel * np.abs(dgs), 1, keepdims=True)
    mag_l = p * dsel + p * S1
    c = 2.0 * (rng_l + E + k + 8) * 2.0 ** -24
    err = np.abs(dl - dl_ref)
    assert np.all(err <= c * mag_l + 1e-37), f"d_logits outside the bound: worst {np.max(err / (c * mag_l + 1e-37))}"
    if w.mode == workloads.TOPK_SOFTMAX:
        assert np.all(dl[~sel] == 0.0), "unselected experts get no gradient in top-k-then-softmax"
    return plan


SMALL = [
    W["tiny"],
    W["v2_top2"].scaled(1000),
    W["fine_shared"].scaled(333),
    W["fp8_skewed"].scaled(1500),
    W["prefill_cap"].scaled(700),
    W["prefill_reassign"].scaled(700),  # re-assigned slots keep their gates and gradients
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_backward_small_exact(w):
    _check_backward(w)


@pytest.mark.parametrize("name", ["v2_top2", "fine_shared", "fp8_skewed", "prefill_cap"])
def test_backward_full_size_sampled(name):
    _check_backward(W[name], token_sample=400)


def _edge(T, H, E, k, P, mode=0, cap=0.0, seed=77, **kw):
    return workloads.Workload(f"bwd_T{T}_H{H}_E{E}_k{k}", T=T, H=H, E=E, k=k, P=P, mode=mode,
                              capacity_factor=cap, seed=seed, **kw)


EDGES = [
    _edge(0, 256, 8, 2, 4),                      # empty batch
    _edge(1, 8, 2, 1, 1),                        # one token, one vector per row
    _edge(97, 4104, 16, 9, 4),                   # ragged rows: three passes, partial tail
    _edge(300, 16384, 16, 2, 4),                 # longest rows: multi-pass dot products
    _edge(129, 512, 256, 16, 8, mode=1),         # E = 256, k = 16 (largest templates)
    _edge(200, 1024, 64, 9, 8, mode=1),          # k > 8: one vector per thread
    _edge(2000, 256, 16, 4, 4, cap=1.25, zipf_bias=True, logit_std=3.0),  # many drops
]


@pytest.mark.parametrize("w", EDGES, ids=[w.name for w in EDGES])
def test_backward_edge_cases(w):
    _check_backward(w)


def test_backward_is_deterministic():
    w = W["fine_shared"].scaled(500)
    inp = workloads.make_inputs(w, "cuda")
    plan, _, _, R, eo, _ = run_gpu(w, inp)
    dy = workloads.make_dy(w, "cuda")
    dp = workloads.make_d_packed(w, max(R, 1), "cuda")
    plan.backward(inp["logits"], dy, eo, dp)
    first = (plan.d_gates.clone(), plan.d_logits.clone(), plan.dx.clone(), plan.d_expert_out[:R].clone())
    plan.backward(inp["logits"], dy, eo, dp)
    again = (plan.d_gates, plan.d_logits, plan.dx, plan.d_expert_out[:R])
    for a, b in zip(first, again):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
