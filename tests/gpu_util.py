"""Helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_moe_gate_warp_gb300 import RoutePlan, RouteShape, workloads


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f_of_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def shape_of(w: workloads.Workload) -> RouteShape:
    return RouteShape(T=w.T, H=w.H, E=w.E, k=w.k, P=w.P, mode=w.mode, fp8=w.fp8, Ks=w.Ks,
                      capacity=w.capacity)


def run_gpu(w: workloads.Workload, inputs: dict, device="cuda"):
    """The four calls on the GPU.  Returns the plan, host snapshots of the
    gate outputs taken before the layout zeroes dropped gates, R, and the
    expert outputs used by the combine."""
    plan = RoutePlan(shape_of(w), device)
    plan.gate(inputs["logits"])
    gates_pre = plan.gates.clone()
    plan.dispatch_layout()
    plan.dispatch(inputs["x"])
    R = int(plan.layout.offsets[w.E].item())
    if w.identity_experts:
        eo = plan.packed
    else:
        eo = workloads.make_expert_out(w, max(R, 1), device)
    plan.combine(eo, inputs["shared"])
    status = plan.status()
    return plan, gates_pre, R, eo, status


def check_gate(w, plan, gates_pre, logits_np, tol_gate=1e-6):
    idx, g64, counts, aux, ent = oracle.gate(logits_np, w.k, w.mode)
    T = w.T
    assert np.array_equal(plan.topk_idx.cpu().numpy()[:T], idx), "topk_idx differs from the oracle"
    assert np.array_equal(plan.expert_counts.cpu().numpy(), counts), "expert_counts differ"
    gerr = np.max(np.abs(gates_pre.cpu().double().numpy()[:T] - g64)) if T else 0.0
    assert gerr <= tol_gate, f"gate error {gerr}"
    # aux: both sides work from the same integer counts in fp64 (bound asked: 1e-6)
    assert abs(plan.aux_loss.item() - aux) <= 1e-9, (plan.aux_loss.item(), aux)
    # entropy: exponent + fp32-mantissa logarithms on the device (~1e-7); bound 1e-6
    assert abs(plan.entropy.item() - ent) <= 1e-6, (plan.entropy.item(), ent)
    return idx, counts


def check_layout(w, plan, idx, gates_pre):
    gpre = gates_pre.cpu().numpy()[:w.T]
    L = oracle.layout(idx, w.E, w.P, w.capacity, gates_f32=gpre)
    lay = plan.layout
    A = w.T * w.k
    assert np.array_equal(lay.counts.cpu().numpy(), L["counts"]), "kept counts"
    assert np.array_equal(lay.offsets.cpu().numpy(), L["offsets"]), "offsets"
    assert np.array_equal(lay.part_rows.cpu().numpy(), L["part_rows"]), "part_rows"
    assert np.array_equal(lay.part_offsets.cpu().numpy(), L["part_offsets"]), "part_offsets"
    assert np.array_equal(lay.part_tokens.cpu().numpy(), L["part_tokens"]), "part_tokens"
    assert int(lay.dropped.item()) == L["dropped"], "dropped"
    if A:
        assert np.array_equal(lay.dst_row.cpu().numpy()[:A], L["dst_row"]), "dst_row"
        assert np.array_equal(lay.capacity_mask.cpu().numpy()[:A], L["capacity_mask"]), "capacity_mask"
        assert np.array_equal(lay.src_pos.cpu().numpy()[:L["R"]], L["src_pos"]), "src_pos"
        # gates after the layout: dropped slots zeroed, others untouched
        assert np.array_equal(plan.gates.cpu().numpy()[:w.T].ravel().view(np.uint32),
                              L["gates"].ravel().view(np.uint32)), "gates after layout"
    return L


def sample_rows(n: int, rng, m: int = 512) -> np.ndarray:
    if n <= 3 * m:
        return np.arange(n, dtype=np.int64)
    pick = np.concatenate([np.arange(64), np.arange(n - 64, n), rng.choice(n, m, replace=False)])
    return np.unique(pick).astype(np.int64)


def check_dispatch(w, plan, L, x_bits, rows):
    if rows.size == 0:
        return
    rows_t = torch.from_numpy(rows).to(plan.packed.device)
    if w.fp8:
        got = plan.packed.index_select(0, rows_t).cpu().numpy()
        got_s = plan.scales.index_select(0, rows_t).cpu().numpy()
        want, want_s = oracle.dispatch_fp8_rows(x_bits, w.k, L["src_pos"], rows)
        assert np.array_equal(got, want), f"fp8 codes differ in {np.sum(np.any(got != want, 1))} rows"
        assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), "fp8 scales differ"
    else:
        got = bits(plan.packed.index_select(0, rows_t))
        want = oracle.dispatch_bf16_rows(x_bits, w.k, L["src_pos"], rows)
        assert np.array_equal(got, want), "packed bf16 rows differ"


def _ulp_bf16(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return 2.0 ** (np.maximum(e, -126) - 7)


def check_combine(w, plan, L, eo, shared, tokens):
    """Bit-exact against the oracle's pinned fp32 order, and within the
    error bound of the fp64 reference; both fed the GPU's fp32 gates and
    the oracle's layout (bit-equal to the GPU's)."""
    if tokens.size == 0:
        return
    T, k = w.T, w.k
    dst = L["dst_row"].reshape(T, k)[tokens]
    need = np.unique(dst[dst >= 0])
    eo_sub = bits(eo.index_select(0, torch.from_numpy(need.astype(np.int64)).to(eo.device))) \
        if need.size else np.zeros((1, w.H), np.uint16)
    remap = np.full(T * k, -1, np.int32)
    flat = (tokens[:, None] * k + np.arange(k)[None, :]).ravel()
    sub = dst.ravel()
    remap[flat] = np.where(sub >= 0, np.searchsorted(need, sub), -1)
    n = tokens.size
    g_c = plan.gates.cpu().numpy()[:T][tokens]
    remap_c = remap.reshape(T, k)[tokens].ravel()
    sh_c = None
    if shared is not None:  # [Ks, T, H] -> [Ks, n, H], tokens renumbered 0..n-1
        sh_c = bits(shared.index_select(1, torch.from_numpy(tokens).to(shared.device)))
    y_ref = oracle.combine_f32order(eo_sub, g_c, remap_c, np.arange(n), n, k, sh_c)
    ref, mag = oracle.combine_ref64(eo_sub, g_c, remap_c, np.arange(n), n, k, sh_c)
    got = bits(plan.y.index_select(0, torch.from_numpy(tokens).to(plan.y.device)))
    assert np.array_equal(got, y_ref), f"combine differs from the pinned fp32 order in {np.sum(got != y_ref)} values"
    err = np.abs(f_of_bits(got).astype(np.float64) - ref)
    n_terms = k + w.Ks
    bound = _ulp_bf16(ref) + n_terms * 2.0 ** -24 * mag
    assert np.all(err <= bound), "combine outside the fp64 error bound"
    within_ulp = float(np.mean(err <= _ulp_bf16(ref)))
    return within_ulp
