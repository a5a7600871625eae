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

import concurrent.futures as cf
import os

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


def oracle_layout(w, og):
    """The oracle's layout of the oracle's gate outputs og."""
    idx, g64 = og[0], og[1]
    if getattr(w, "reassign", False) and w.capacity > 0:
        return oracle.layout_reassign(idx, w.E, w.P, w.capacity, gates_f32=g64.astype(np.float32))
    return oracle.layout(idx, w.E, w.P, w.capacity, gates_f32=g64.astype(np.float32))


def route_with_oracle(w, plan, logits: torch.Tensor):
    """moe_route on the GPU (gate and layout in one launch), the oracle's
    gate and layout on the same logits, then the oracle's fp32 gates (zero
    at dropped slots) written into the plan for the calls that follow.
    Returns (GPU gates as the call left them, oracle gate outputs)."""
    assert plan.fused_route, "moe_route is not used for this shape"
    plan.route(logits)
    gates_pre = plan.gates.clone()
    og = oracle.gate(logits.cpu().numpy(), w.k, w.mode)
    if w.T:
        L = oracle_layout(w, og)
        plan.gates[:w.T].copy_(torch.from_numpy(L["gates"]).to(plan.gates.device))
    return gates_pre, og


def run_gpu(w: workloads.Workload, inputs: dict, device="cuda", fused=None):
    """The path on the GPU (outputs poisoned first): moe_route (or, with
    fused=False or re-assigned overflow, moe_gate + the layout call), then
    dispatch and combine.  Returns the plan, the GPU's gate weights, the
    oracle's gate outputs, R, the expert outputs used by the combine and the
    device status."""
    plan = RoutePlan(shape_of(w), device)
    poison(plan)
    if fused is None:
        fused = plan.fused_route
    if fused:
        gates_pre, og = route_with_oracle(w, plan, inputs["logits"])
    else:
        plan.fused_route = False
        gates_pre, og = gate_with_oracle(w, plan, inputs["logits"])
        plan.dispatch_layout()
    plan.dispatch(inputs["x"])
    R = int(plan.layout.offsets[w.E].item())
    if w.identity_experts:
        eo = plan.packed
    else:
        eo = workloads.make_expert_out(w, max(plan.r_max, 1), device)
    if w.fp8_combine:
        plan.quantize_expert_out(eo)
        plan.combine_fp8(inputs["shared"])
    else:
        plan.combine(eo, inputs["shared"])
    status = plan.status()
    return plan, gates_pre, og, R, eo, status


def check_gate(w, plan, gates_pre, og, tol_gate=1e-6):
    """The gate's outputs against the oracle's.  After moe_route the slots
    the layout dropped hold exactly 0 (the layout's capacity_mask, itself
    compared bit for bit by check_layout, says which)."""
    idx, g64, counts, aux, ent = og
    T = w.T
    assert np.array_equal(plan.topk_idx.cpu().numpy()[:T], idx), "topk_idx differs from the oracle"
    assert np.array_equal(plan.expert_counts.cpu().numpy(), counts), "expert_counts differ"
    gp = gates_pre.cpu().double().numpy()[:T]
    if plan.fused_route and T:
        dropped = plan.layout.capacity_mask.cpu().numpy()[:T * w.k].reshape(T, w.k) == 0
        assert np.all(gp[dropped] == 0.0), "moe_route must zero the gates of dropped slots"
        gp = np.where(dropped, g64, gp)
    gerr = np.max(np.abs(gp - g64)) if T else 0.0
    assert gerr <= tol_gate, f"gate error {gerr}"
    # aux: both sides work from the same integer counts in fp64 (bound asked: 1e-6)
    assert abs(plan.aux_loss.item() - aux) <= 1e-9, (plan.aux_loss.item(), aux)
    # entropy: exponent + fp32-mantissa logarithms on the device (~1e-7); bound 1e-6
    assert abs(plan.entropy.item() - ent) <= 1e-6, (plan.entropy.item(), ent)
    return idx, counts


def check_layout(w, plan, og):
    """The GPU layout against the oracle's (the plan's gates are the
    oracle's: swapped in before the layout call, or after moe_route)."""
    L = oracle_layout(w, og)
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


# --- full comparisons: chunks of rows / tokens, the oracle over a thread pool
# (its C calls release the interpreter lock, and so do numpy's large array ops)
_POOL = None


def pool():
    global _POOL
    if _POOL is None:
        n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        _POOL = cf.ThreadPoolExecutor(max_workers=max(1, min(16, n)))
    return _POOL


def split(a: np.ndarray, parts: int):
    """Contiguous pieces of index array `a` (empty pieces dropped)."""
    if a.size == 0:
        return []
    edges = np.linspace(0, a.size, max(1, min(parts, a.size)) + 1).astype(np.int64)
    return [a[edges[i]:edges[i + 1]] for i in range(len(edges) - 1) if edges[i + 1] > edges[i]]


def pmap(fn, pieces):
    return list(pool().map(fn, pieces))


def chunks(n: int, size: int):
    for a in range(0, n, size):
        yield np.arange(a, min(n, a + size), dtype=np.int64)


class FP8Ref:
    """The oracle's FP8 codes and scales of packed rows for one quantiser
    mode; for the grouped modes the group extremes are taken once over
    every row (src_row_all[r] = source row of packed row r)."""

    def __init__(self, mode, src_bits, src_row_all, offsets):
        self.mode, self.src, self.src_row = int(mode), src_bits, src_row_all
        if self.mode != oracle.FP8_PER_TOKEN:
            self.group, ng = oracle.row_groups(self.mode, offsets, np.arange(src_row_all.size))
            self.params = oracle.fp8_group_params(src_bits, src_row_all, self.group, ng)

    def _rows(self, rows):
        if self.mode == oracle.FP8_PER_TOKEN:
            return oracle.quantize_rows_grouped(self.src, self.src_row[rows], np.arange(rows.size, dtype=np.int32),
                                                rows.size)
        return oracle.quantize_rows_with_params(self.src, self.src_row[rows], self.group[rows], self.params)

    def rows(self, rows):
        parts = pmap(self._rows, split(rows, 16))
        if not parts:
            return np.zeros((0, self.src.shape[1]), np.uint8), np.zeros((0, 2), np.float32)
        return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def oracle_fp8_rows(mode, src_bits, src_row_all, offsets, rows):
    """The oracle's codes and scales of packed rows `rows` for a quantiser
    mode: group extremes over every row, then the listed rows encoded."""
    return FP8Ref(mode, src_bits, src_row_all, offsets).rows(rows)


def check_dispatch(w, plan, L, x_bits, rows, fp8ref=None):
    if rows.size == 0:
        return
    contiguous = rows[-1] - rows[0] + 1 == rows.size
    if contiguous:
        dev = plan.packed[int(rows[0]):int(rows[-1]) + 1]
    else:
        dev = plan.packed.index_select(0, torch.from_numpy(rows).to(plan.packed.device))
    if w.fp8:
        got = dev.cpu().numpy()
        sc = plan.scales[int(rows[0]):int(rows[-1]) + 1] if contiguous else \
            plan.scales.index_select(0, torch.from_numpy(rows).to(plan.scales.device))
        got_s = sc.cpu().numpy()
        if fp8ref is None:
            fp8ref = FP8Ref(int(w.fp8), x_bits, L["src_pos"].astype(np.int64) // w.k, L["offsets"])
        want, want_s = fp8ref.rows(rows)
        assert np.array_equal(got, want), f"fp8 codes differ in {np.sum(np.any(got != want, 1))} rows"
        assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), "fp8 scales differ"
    else:
        got = bits(dev)
        want = np.concatenate(pmap(lambda r: oracle.dispatch_bf16_rows(x_bits, w.k, L["src_pos"], r),
                                   split(rows, 16)))
        assert np.array_equal(got, want), f"packed bf16 rows differ in {np.sum(np.any(got != want, 1))} rows"


def check_dispatch_full(w, plan, L, x_bits, chunk=1 << 15):
    """Every packed row (codes and scale words for FP8), in chunks."""
    fp8ref = None
    if w.fp8:
        fp8ref = FP8Ref(int(w.fp8), x_bits, L["src_pos"].astype(np.int64) // w.k, L["offsets"])
    for rows in chunks(L["R"], chunk):
        check_dispatch(w, plan, L, x_bits, rows, fp8ref)


def _ulp_bf16(v):
    """One bf16 ulp at |v|: 2^(floor(log2|v|) - 7), the exponent read from the
    fp64 bits (exact), at least the subnormal step 2^-133."""
    e = ((np.ascontiguousarray(v, np.float64).view(np.uint64) >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64)
    return np.ldexp(1.0, np.maximum(e - 1023, -126) - 7)


def oracle_expert_rows(w, L, eo, x_bits, need):
    """bf16 bits of expert-output rows `need` as the oracle sees them: the
    seeded tensor, or, for identity experts, the oracle's own dispatch."""
    if need.size == 0:
        return np.zeros((1, w.H), np.uint16)
    if w.identity_experts:
        return oracle.dispatch_bf16_rows(x_bits, w.k, L["src_pos"], need)
    return bits(eo.index_select(0, torch.from_numpy(need.astype(np.int64)).to(eo.device)))


class UlpStats:
    """Combine outputs against the fp64 reference: how many lie beyond one
    bf16 ulp of it (each then excused by the fp32 summation allowance
    n * 2^-24 * sum|terms|), and the largest share of that allowance used."""

    def __init__(self):
        self.outputs = 0
        self.beyond_ulp = 0
        self.max_allowance_used = 0.0

    def add(self, outputs, beyond, used):
        self.outputs += outputs
        self.beyond_ulp += beyond
        self.max_allowance_used = max(self.max_allowance_used, used)

    def merge(self, o):
        self.add(o.outputs, o.beyond_ulp, o.max_allowance_used)

    def as_dict(self):
        return {"outputs": self.outputs, "beyond_1ulp": self.beyond_ulp,
                "max_allowance_used": self.max_allowance_used}


ULP_RECORDS = []  # (workload, UlpStats) of every full comparison, printed by the session summary


def _compare_combine_part(got, y_ref, ref, mag, n_terms):
    """One piece of a combine comparison: bit-exact against the pinned fp32
    order, within the fp64 bound; returns (mismatches, outside bound,
    outputs beyond 1 ulp, largest allowance share used)."""
    mism = int(np.count_nonzero(got != y_ref))
    err = np.abs(f_of_bits(got).astype(np.float64) - ref)
    ulp = _ulp_bf16(ref)
    allow = n_terms * 2.0 ** -24 * mag
    out = int(np.count_nonzero(err > ulp + allow))
    over = err > ulp
    beyond = int(np.count_nonzero(over))
    used = float(np.max((err[over] - ulp[over]) / np.maximum(allow[over], 1e-300))) if beyond else 0.0
    return mism, out, beyond, used


def check_combine(w, plan, L, eo, shared, tokens, x_bits=None, fp8ref=None, stats=None):
    """Bit-exact against the oracle's pinned fp32 order, and within the
    error bound of the fp64 reference, both sides fed the oracle's gates
    and layout and the seeded expert outputs.  Returns (and adds to
    `stats`) the count of outputs beyond one bf16 ulp of the reference."""
    st = UlpStats() if stats is None else stats
    if tokens.size == 0:
        return st
    T, k = w.T, w.k
    dst = L["dst_row"].reshape(T, k)[tokens]
    need = np.unique(dst[dst >= 0])
    n = tokens.size
    remap_c = np.where(dst >= 0, np.searchsorted(need, np.maximum(dst, 0)), -1).astype(np.int32).ravel()
    g_c = np.ascontiguousarray(L["gates"][tokens])
    sh_c = None
    if shared is not None:  # [Ks, T, H] -> [Ks, n, H], tokens renumbered 0..n-1
        sh_c = bits(shared.index_select(1, torch.from_numpy(tokens).to(shared.device)))
    got = bits(plan.y.index_select(0, torch.from_numpy(tokens).to(plan.y.device)))
    n_terms = k + w.Ks
    if w.fp8_combine:
        if fp8ref is None:
            R = L["R"]
            fp8ref = FP8Ref(int(w.fp8_combine), oracle_expert_rows(w, L, eo, x_bits, np.arange(R)),
                            np.arange(R, dtype=np.int64), L["offsets"])
        if need.size:
            codes, scales = fp8ref.rows(need)
            need_t = torch.from_numpy(need.astype(np.int64)).to(plan.eo_codes.device)
            assert np.array_equal(plan.eo_codes.index_select(0, need_t).cpu().numpy(), codes), \
                "expert-output FP8 codes differ"
            assert np.array_equal(plan.eo_scales.index_select(0, need_t).cpu().numpy().view(np.uint32),
                                  scales.view(np.uint32)), "expert-output FP8 scales differ"
        else:
            codes, scales = np.zeros((1, w.H), np.uint8), np.zeros((1, 2), np.float32)
        n_terms += 1  # the dequantisation rounding

        def part(idx):
            ys = oracle.combine_fp8_f32order(codes, scales, g_c, remap_c, idx, n, k, sh_c)
            ref, mag = oracle.combine_fp8_ref64(codes, scales, g_c, remap_c, idx, n, k, sh_c)
            return _compare_combine_part(got[idx], ys, ref, mag, n_terms)
    else:
        eo_sub = oracle_expert_rows(w, L, eo, x_bits, need)

        def part(idx):
            ys = oracle.combine_f32order(eo_sub, g_c, remap_c, idx, n, k, sh_c)
            ref, mag = oracle.combine_ref64(eo_sub, g_c, remap_c, idx, n, k, sh_c)
            return _compare_combine_part(got[idx], ys, ref, mag, n_terms)

    res = pmap(part, split(np.arange(n, dtype=np.int64), 16))
    mism = sum(r[0] for r in res)
    assert mism == 0, f"combine differs from the pinned fp32 order in {mism} values"
    out = sum(r[1] for r in res)
    assert out == 0, f"combine outside the fp64 error bound in {out} values"
    st.add(n * w.H, sum(r[2] for r in res), max(r[3] for r in res))
    return st


def check_combine_full(w, plan, L, eo, shared, x_bits=None, chunk=None):
    """Every token's output row, in chunks of tokens; records and returns
    the beyond-one-ulp statistics."""
    if chunk is None:  # about 64 MB of expert rows per chunk
        chunk = max(256, (1 << 25) // max(1, w.k * w.H))
    fp8ref = None
    if w.fp8_combine and L["R"]:
        R = L["R"]
        fp8ref = FP8Ref(int(w.fp8_combine), oracle_expert_rows(w, L, eo, x_bits, np.arange(R)),
                        np.arange(R, dtype=np.int64), L["offsets"])
    st = UlpStats()
    for toks in chunks(w.T, chunk):
        check_combine(w, plan, L, eo, shared, toks, x_bits, fp8ref, st)
    ULP_RECORDS.append((w.name, st))
    return st


def route_checked(w, plan, logits):
    """Routing on an existing plan (moe_route when the plan uses it, else
    gate then layout), compared with the oracle, the oracle's gates swapped
    in; returns the oracle layout."""
    if plan.fused_route:
        gates_pre, og = route_with_oracle(w, plan, logits)
    else:
        gates_pre, og = gate_with_oracle(w, plan, logits)
        plan.dispatch_layout()
    assert plan.status() == 0
    check_gate(w, plan, gates_pre, og)
    return check_layout(w, plan, og)


__all__ = ["bits", "f_of_bits", "shape_of", "gate_with_oracle", "route_with_oracle", "oracle_layout", "run_gpu", "check_gate", "check_layout",
           "sample_rows", "oracle_fp8_rows", "FP8Ref", "check_dispatch", "check_dispatch_full", "oracle_expert_rows",
           "check_combine", "check_combine_full", "UlpStats", "ULP_RECORDS", "route_checked", "abi", "poison",
           "pool", "pmap", "split", "chunks"]
