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
from gpu_util import bits, check_gate, check_layout, chunks, f_of_bits, pmap, run_gpu, split

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


def _check_backward(w, seed=11):
    """Forward on the GPU (gate compared, oracle gates swapped in, layout
    compared), then the backward calls on seeded gradients; the oracle gets
    its own layout and gates and the same seeded tensors.  Every token is
    compared, in chunks of tokens over a thread pool."""
    inp = workloads.make_inputs(w, "cuda")
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp)
    assert status == 0
    check_gate(w, plan, gates_pre, og)
    L = check_layout(w, plan, og)
    dy = workloads.make_dy(w, "cuda")
    dp = workloads.make_d_packed(w, max(plan.r_max, 1), "cuda")
    dg_in = workloads.make_d_gates(w, "cuda")
    plan.combine_backward(dy, eo)
    plan.gate_backward(inp["logits"], dg_in)
    plan.dispatch_backward(dp)
    assert plan.status() == 0, "device status after the backward"
    T, k, H = w.T, w.k, w.H
    if T == 0:
        return plan
    x_bits = bits(inp["x"]) if w.identity_experts else None
    logits_all = inp["logits"].cpu().numpy()
    dg_all = plan.d_gates.cpu().numpy()[:T]
    dgs_all = dg_in.cpu().numpy()[:T].astype(np.float64)
    dl_all = plan.d_logits.cpu().numpy()[:T].astype(np.float64)
    chunk = max(64, (1 << 25) // max(1, k * H))  # ~32 M expert-row values per chunk
    for toks in chunks(T, chunk):
        # the rows a chunk needs come off the device on this thread; the
        # oracle and the comparisons run on the pool
        dst = L["dst_row"].reshape(T, k)[toks]
        need = np.unique(dst[dst >= 0])
        eo_rows = _gather(eo, need) if not w.identity_experts else \
            (oracle.dispatch_bf16_rows(x_bits, k, L["src_pos"], need) if need.size else _gather(eo, need))
        got = dict(dy=_gather(dy, toks), d_eo=_gather(plan.d_expert_out, need), dp=_gather(dp, need),
                   dx=_gather(plan.dx, toks))
        errs = pmap(lambda sub: _check_backward_tokens(w, L, og, toks, sub, dst, need, eo_rows, got, dg_all,
                                                       logits_all, dgs_all, dl_all),
                    split(np.arange(toks.size, dtype=np.int64), 8))
        errs = [e for e in errs if e]
        assert not errs, errs[0]
    return plan


def _check_backward_tokens(w, L, og, toks, sub, dst, need, eo_rows, got, dg_all, logits_all, dgs_all, dl_all):
    """The backward checks for tokens toks[sub]; returns an error message or
    None (assertion messages do not cross the thread pool well)."""
    T, k, H, E = w.T, w.k, w.H, w.E
    t_ids = toks[sub]
    n = t_ids.size
    d = dst[sub]
    remap = np.where(d >= 0, np.searchsorted(need, np.maximum(d, 0)), -1).astype(np.int32).ravel()
    dy_c = got["dy"][sub]
    g_c = np.ascontiguousarray(L["gates"][t_ids])
    # combine backward
    d_eo_ref, dg_ref = oracle.combine_backward(dy_c, eo_rows, g_c, remap, np.arange(n), k)
    kept = remap >= 0
    if not np.array_equal(got["d_eo"][remap[kept]], d_eo_ref[kept]):
        return "d_expert_out differs from the oracle"
    dg = dg_all[t_ids]
    if not np.all(dg.ravel()[~kept] == 0.0):
        return "dropped slots must get a zero gate gradient"
    dyf = np.abs(f_of_bits(dy_c).astype(np.float64))
    mag = np.zeros(n * k)
    for j in range(k):
        kj = remap[j::k] >= 0
        if kj.any():
            eo_abs = np.abs(f_of_bits(eo_rows[remap[j::k][kj]]).astype(np.float64))
            mag[j::k][kj] = np.einsum("ih,ih->i", dyf[kj], eo_abs)
    bound = (H / 256 + 14) * 2.0 ** -24 * mag + 1e-30
    err = np.abs(dg.ravel().astype(np.float64) - dg_ref.ravel())
    if not np.all(err <= bound):
        return f"d_gates outside the fp32 bound: worst {np.max(err / bound)} x bound"
    # dispatch backward
    dx_ref, dx64 = oracle.dispatch_backward(got["dp"], remap, np.arange(n), k)
    dx = got["dx"][sub]
    if not np.array_equal(dx, dx_ref):
        return f"dx differs from the oracle in {np.sum(dx != dx_ref)} values"
    none_kept = ~kept.reshape(n, k).any(1)
    if np.any(dx[none_kept]):
        return "a token with no kept slot has dx = 0"
    # gate backward on the seeded gate gradients
    logits = logits_all[t_ids]
    idx = og[0][t_ids]
    dgs = dgs_all[t_ids]
    dl_ref = oracle.gate_backward(logits, idx, dgs, w.mode)
    dl = dl_all[t_ids]
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
    if not np.all(err <= c * mag_l + 1e-37):
        return f"d_logits outside the bound: worst {np.max(err / (c * mag_l + 1e-37))}"
    if w.mode == workloads.TOPK_SOFTMAX and not np.all(dl[~sel] == 0.0):
        return "unselected experts get no gradient in top-k-then-softmax"
    return None


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
def test_backward_full_size(name):
    _check_backward(W[name])


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
    dp = workloads.make_d_packed(w, max(plan.r_max, 1), "cuda")
    plan.backward(inp["logits"], dy, eo, dp)
    first = (plan.d_gates.clone(), plan.d_logits.clone(), plan.dx.clone(), plan.d_expert_out[:R].clone())
    plan.backward(inp["logits"], dy, eo, dp)
    again = (plan.d_gates, plan.d_logits, plan.dx, plan.d_expert_out[:R])
    for a, b in zip(first, again):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
