"""GPU: the step captured as a CUDA graph (RouteGraph) and replayed, against
the oracle on the same seeded inputs, for two input batches replayed through
the same graph (the graph must read its buffers, not captured values)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import RouteGraph, workloads
from gpu_util import bits, check_dispatch, shape_of

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()
    torch.cuda.init()


def _check_replay(w, g, inp, eo):
    """Gate within 1e-6 of the oracle's fp64 gates, ids and layout bit-exact,
    dispatch bit-exact; returns the oracle layout."""
    plan = g.step(inp["logits"], inp["x"], eo, inp["shared"])
    torch.cuda.synchronize()
    assert g.status() == 0
    og = oracle.gate(inp["logits"].cpu().numpy(), w.k, w.mode)
    assert np.array_equal(plan.topk_idx[:w.T].cpu().numpy(), og[0])
    assert np.array_equal(plan.expert_counts.cpu().numpy(), og[2])
    L = oracle.layout(og[0], w.E, w.P, w.capacity, gates_f32=og[1].astype(np.float32))
    # gates after the layout: the gate's weights where kept, 0 where dropped
    kept = L["capacity_mask"].reshape(w.T, w.k) != 0
    g_gpu = plan.gates[:w.T].cpu().double().numpy()
    gerr = np.max(np.abs(g_gpu - og[1])[kept]) if kept.any() else 0.0
    assert gerr <= 1e-6, f"gate error {gerr}"
    assert np.all(g_gpu[~kept] == 0.0)
    lay = plan.layout
    assert np.array_equal(lay.offsets.cpu().numpy(), L["offsets"])
    assert np.array_equal(lay.dst_row.cpu().numpy()[:w.T * w.k], L["dst_row"])
    assert np.array_equal(lay.src_pos.cpu().numpy()[:L["R"]], L["src_pos"][:L["R"]])
    check_dispatch(w, plan, L, bits(inp["x"]), np.arange(L["R"], dtype=np.int64))
    return plan, L


def test_identity_experts_return_x():
    """tiny: identity experts and gates summing to 1 give y == x bit for
    bit, whatever the gates' last-bit rounding."""
    w = W["tiny"]
    g = RouteGraph(shape_of(w), "cuda")
    for seed in (w.seed, w.seed + 1):
        wb = workloads.Workload(**{**w.__dict__, "seed": seed})
        inp = workloads.make_inputs(wb, "cuda")
        # identity experts: the expert outputs are the packed rows of this batch
        plan, L = _check_replay(wb, g, inp, None)
        g.step(expert_out=plan.packed[:L["R"]].clone())
        torch.cuda.synchronize()
        assert np.array_equal(bits(plan.y[:w.T]), bits(inp["x"]))


@pytest.mark.parametrize("name,T", [("v2_top2", 1000), ("fine_shared", 333), ("prefill_cap", 700)])
def test_replay_matches_oracle(name, T):
    """Seeded expert outputs: the combine within the fp64 reference bound
    (the graph's combine uses its own gates, which the oracle does not
    take as input)."""
    w = W[name].scaled(T)
    g = RouteGraph(shape_of(w), "cuda")
    for seed in (w.seed, w.seed + 5):
        wb = workloads.Workload(**{**w.__dict__, "seed": seed})
        inp = workloads.make_inputs(wb, "cuda")
        L0 = oracle.layout(oracle.gate(inp["logits"].cpu().numpy(), w.k, w.mode)[0], w.E, w.P, w.capacity)
        eo = workloads.make_expert_out(wb, max(int(L0["R"]), 1), "cuda")
        plan, L = _check_replay(wb, g, inp, eo)
        g_or = L["gates"]  # the oracle's fp32 gates after the layout (dropped slots zeroed)
        T_, k = w.T, w.k
        eo_bits = bits(eo[:max(L["R"], 1)])
        sh = None if inp["shared"] is None else bits(inp["shared"])
        dst = L["dst_row"].astype(np.int32)
        ref, mag = oracle.combine_ref64(eo_bits, g_or, dst, np.arange(T_), T_, k, sh)
        _, mag1 = oracle.combine_ref64(eo_bits, np.ones_like(g_or), dst, np.arange(T_), T_, k, sh)
        y = plan.y[:T_].float().cpu().numpy().astype(np.float64)
        a = np.abs(ref)
        e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
        ulp = 2.0 ** (np.maximum(e, -126) - 7)
        # one bf16 ulp, the fp32 summation bound, and the GPU's gates (each
        # within 1e-6 of the oracle's) times the sum of |expert outputs|
        bound = ulp + (k + w.Ks) * 2.0 ** -24 * mag + 1e-6 * mag1
        assert np.all(np.abs(y - ref) <= bound), f"{np.sum(np.abs(y - ref) > bound)} values outside the bound"


@pytest.mark.parametrize("name,T,variant", [("fp8_skewed", 1500, {}), ("prefill_reassign", 700, {}),
                                             ("fp8_skewed", 1200, {"fp8": 3, "fp8_combine": 2})])
def test_replay_fp8_and_reassign(name, T, variant):
    """FP8 dispatch (per token; global codes with FP8 expert outputs) and
    the re-assigning layout through the graph: ids, counts, layout and
    packed rows (codes and scales) against the oracle."""
    w = workloads.Workload(**{**W[name].scaled(T).__dict__, **variant})
    g = RouteGraph(shape_of(w), "cuda")
    for seed in (w.seed, w.seed + 3):
        wb = workloads.Workload(**{**w.__dict__, "seed": seed})
        inp = workloads.make_inputs(wb, "cuda")
        plan = g.step(inp["logits"], inp["x"], None, inp["shared"])
        torch.cuda.synchronize()
        assert g.status() == 0
        og = oracle.gate(inp["logits"].cpu().numpy(), w.k, w.mode)
        assert np.array_equal(plan.topk_idx[:w.T].cpu().numpy(), og[0])
        g32 = og[1].astype(np.float32)
        L = (oracle.layout_reassign(og[0], w.E, w.P, w.capacity, gates_f32=g32) if w.reassign
             else oracle.layout(og[0], w.E, w.P, w.capacity, gates_f32=g32))
        assert np.array_equal(plan.layout.offsets.cpu().numpy(), L["offsets"])
        assert np.array_equal(plan.layout.dst_row.cpu().numpy()[:w.T * w.k], L["dst_row"])
        check_dispatch(w, plan, L, bits(inp["x"]), np.arange(L["R"], dtype=np.int64))


def test_empty_batch_graph():
    w = W["v2_top2"].scaled(0)
    g = RouteGraph(shape_of(w), "cuda")
    g.step()
    torch.cuda.synchronize()
    assert g.status() == 0
