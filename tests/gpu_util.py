"""Helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, and compare.

Every oracle input is either a seeded input (from `workloads`) or an oracle
output; nothing the CUDA path computed is fed to the oracle.  Where a later
call of the path consumes an earlier call's result (the combine reads the
gate weights), the test hands that call the oracle's value instead, so both
sides start from the same bits: after the gate has been compared, the
oracle's fp32 gate weights replace the GPU's in the plan before the layout
runs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_moe_gate_warp_gb300 import RoutePlan, RouteShape, abi, workloads


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f_of_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def shape_of(w: workloads.Workload) -> RouteShape:
    return RouteShape(T=w.T, H=w.H, E=w.E, k=w.k, P=w.P, mode=w.mode, fp8=int(w.fp8), Ks=w.Ks,
                      capacity=w.capacity, fp8_combine=int(w.fp8_combine),
                      reassign=bool(getattr(w, "reassign", False)))


def gate_with_oracle(w, plan, logits: torch.Tensor):
    """moe_gate on the GPU, the oracle's gate on the same logits, then the
    oracle's fp32 gates written into the plan for the calls that follow.
    Returns (GPU gates before the swap, oracle (idx, g64, counts, aux, ent))."""
    plan.gate(logits)
    gates_pre = plan.gates.clone()
    og = oracle.gate(logits.cpu().numpy(), w.k, w.mode)
    if w.T:
        plan.gates[:w.T].copy_(torch.from_numpy(og[1].astype(np.float32)).to(plan.gates.device))
    return gates_pre, og


def poison(plan):
    """Fill every output buffer of a plan with 0xFF bytes, so that a row or
    entry the path fails to write cannot match the oracle by accident."""
    bufs = [plan.topk_idx, plan.gates, plan.expert_counts, plan.aux_loss, plan.entropy, plan.packed, plan.y]
    lay = plan.layout
    bufs += [lay.counts, lay.offsets, lay.part_rows, lay.part_offsets, lay.part_tokens, lay.src_pos, lay.dst_row,
             lay.capacity_mask, lay.dropped]
    for name in ("scales", "eo_codes", "eo_scales"):
        t = getattr(plan, name, None)
        if t is not None:
            bufs.append(t)
    for t in bufs:
        t.view(torch.uint8).fill_(0xFF)


def run_gpu(w: workloads.Workload, inputs: dict, device="cuda"):
    """The path on the GPU (outputs poisoned first).  Returns the plan, the
    GPU's gate weights, the oracle's gate outputs, R, the expert outputs used
    by the combine and the device status."""
    plan = RoutePlan(shape_of(w), device)
    poison(plan)
    gates_pre, og = gate_with_oracle(w, plan, inputs["logits"])
    plan.dispatch_layout()
    plan.dispatch(inputs["x"])
    R = int(plan.layout.offsets[w.E].item())
    if w.identity_experts:
        eo = plan.packed
    else:
        eo = workloads.make_expert_out(w, max(R, 1), device)
    if w.fp8_combine:
        plan.quantize_expert_out(eo)
        plan.combine_fp8(inputs["shared"])
    else:
        plan.combine(eo, inputs["shared"])
    status = plan.status()
    return plan, gates_pre, og, R, eo, status


def check_gate(w, plan, gates_pre, og, tol_gate=1e-6):
    idx, g64, counts, aux, ent = og
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


def check_layout(w, plan, og):
    """The GPU layout (run on the oracle's gates) against the oracle's."""
    idx, g64 = og[0], og[1]
    if getattr(w, "reassign", False) and w.capacity > 0:
        L = oracle.layout_reassign(idx, w.E, w.P, w.capacity, gates_f32=g64.astype(np.float32))
    else:
        L = oracle.layout(idx, w.E, w.P, w.capacity, gates_f32=g64.astype(np.float32))
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


def oracle_fp8_rows(mode, src_bits, src_row_all, offsets, rows):
    """The oracle's codes and scales of packed rows `rows` for a quantiser
    mode: group extremes over every row (src_row_all[r] = source row of
    packed row r), then the listed rows encoded."""
    R = src_row_all.size
    if mode == oracle.FP8_PER_TOKEN:
        return oracle.quantize_rows_grouped(src_bits, src_row_all[rows], np.arange(rows.size, dtype=np.int32),
                                            rows.size)
    group_all, ng = oracle.row_groups(mode, offsets, np.arange(R))
    params = oracle.fp8_group_params(src_bits, src_row_all, group_all, ng)
    return oracle.quantize_rows_with_params(src_bits, src_row_all[rows], group_all[rows], params)


def check_dispatch(w, plan, L, x_bits, rows):
    if rows.size == 0:
        return
    rows_t = torch.from_numpy(rows).to(plan.packed.device)
    if w.fp8:
        got = plan.packed.index_select(0, rows_t).cpu().numpy()
        got_s = plan.scales.index_select(0, rows_t).cpu().numpy()
        if int(w.fp8) == oracle.FP8_PER_TOKEN:
            want, want_s = oracle.dispatch_fp8_rows(x_bits, w.k, L["src_pos"], rows)
        else:
            src_row_all = (L["src_pos"].astype(np.int64) // w.k)
            want, want_s = oracle_fp8_rows(int(w.fp8), x_bits, src_row_all, L["offsets"], rows)
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


def oracle_expert_rows(w, L, eo, x_bits, need):
    """bf16 bits of expert-output rows `need` as the oracle sees them: the
    seeded tensor, or, for identity experts, the oracle's own dispatch."""
    if need.size == 0:
        return np.zeros((1, w.H), np.uint16)
    if w.identity_experts:
        return oracle.dispatch_bf16_rows(x_bits, w.k, L["src_pos"], need)
    return bits(eo.index_select(0, torch.from_numpy(need.astype(np.int64)).to(eo.device)))


def check_combine(w, plan, L, eo, shared, tokens, x_bits=None):
    """Bit-exact against the oracle's pinned fp32 order, and within the
    error bound of the fp64 reference, both sides fed the oracle's gates
    and layout and the seeded expert outputs."""
    if tokens.size == 0:
        return
    T, k = w.T, w.k
    dst = L["dst_row"].reshape(T, k)[tokens]
    need = np.unique(dst[dst >= 0])
    remap = np.full(T * k, -1, np.int32)
    flat = (tokens[:, None] * k + np.arange(k)[None, :]).ravel()
    sub = dst.ravel()
    remap[flat] = np.where(sub >= 0, np.searchsorted(need, sub), -1)
    n = tokens.size
    g_c = L["gates"][tokens]
    remap_c = remap.reshape(T, k)[tokens].ravel()
    sh_c = None
    if shared is not None:  # [Ks, T, H] -> [Ks, n, H], tokens renumbered 0..n-1
        sh_c = bits(shared.index_select(1, torch.from_numpy(tokens).to(shared.device)))
    got = bits(plan.y.index_select(0, torch.from_numpy(tokens).to(plan.y.device)))
    n_terms = k + w.Ks
    if w.fp8_combine:
        R = L["R"]
        mode = int(w.fp8_combine)
        if mode == oracle.FP8_PER_TOKEN:
            eo_sub = oracle_expert_rows(w, L, eo, x_bits, need)
            codes, scales = oracle.quantize_rows_grouped(eo_sub, np.arange(need.size), np.arange(need.size,
                                                         dtype=np.int32), need.size)
        else:
            eo_all = oracle_expert_rows(w, L, eo, x_bits, np.arange(R))
            codes, scales = oracle_fp8_rows(mode, eo_all, np.arange(R, dtype=np.int64), L["offsets"], need)
        if need.size:
            need_t = torch.from_numpy(need.astype(np.int64)).to(plan.eo_codes.device)
            assert np.array_equal(plan.eo_codes.index_select(0, need_t).cpu().numpy(), codes), \
                "expert-output FP8 codes differ"
            assert np.array_equal(plan.eo_scales.index_select(0, need_t).cpu().numpy().view(np.uint32),
                                  scales.view(np.uint32)), "expert-output FP8 scales differ"
        else:
            codes, scales = np.zeros((1, w.H), np.uint8), np.zeros((1, 2), np.float32)
        y_ref = oracle.combine_fp8_f32order(codes, scales, g_c, remap_c, np.arange(n), n, k, sh_c)
        ref, mag = oracle.combine_fp8_ref64(codes, scales, g_c, remap_c, np.arange(n), n, k, sh_c)
        n_terms += 1  # the dequantisation rounding
    else:
        eo_sub = oracle_expert_rows(w, L, eo, x_bits, need)
        y_ref = oracle.combine_f32order(eo_sub, g_c, remap_c, np.arange(n), n, k, sh_c)
        ref, mag = oracle.combine_ref64(eo_sub, g_c, remap_c, np.arange(n), n, k, sh_c)
    assert np.array_equal(got, y_ref), f"combine differs from the pinned fp32 order in {np.sum(got != y_ref)} values"
    err = np.abs(f_of_bits(got).astype(np.float64) - ref)
    bound = _ulp_bf16(ref) + n_terms * 2.0 ** -24 * mag
    assert np.all(err <= bound), "combine outside the fp64 error bound"
    within_ulp = float(np.mean(err <= _ulp_bf16(ref)))
    return within_ulp


def route_checked(w, plan, logits):
    """Gate (compared, then the oracle's gates swapped in) and layout
    (compared) on an existing plan; returns the oracle layout."""
    gates_pre, og = gate_with_oracle(w, plan, logits)
    plan.dispatch_layout()
    assert plan.status() == 0
    check_gate(w, plan, gates_pre, og)
    return check_layout(w, plan, og)


__all__ = ["bits", "f_of_bits", "shape_of", "gate_with_oracle", "run_gpu", "check_gate", "check_layout",
           "sample_rows", "oracle_fp8_rows", "check_dispatch", "oracle_expert_rows", "check_combine",
           "route_checked", "abi", "poison"]
