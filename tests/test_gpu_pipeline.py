"""RoutePipeline (routing of batch i on its own stream, overlapping the
dispatch and combine of batch i-1) gives, batch by batch, the same bits as
the calls run one after another on one stream, and every batch matches the
oracle's combine."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import RoutePipeline, RoutePlan, workloads
from gpu_util import bits, shape_of

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()
    torch.cuda.init()


@pytest.mark.parametrize("w", [W["v2_top2"].scaled(2000), W["fine_shared"].scaled(700),
                               W["fp8_both"].scaled(900), W["prefill_cap"].scaled(1100), W["tiny"]],
                         ids=lambda w: w.name)
def test_pipeline_matches_serial_calls(w):
    batches = []
    for b in range(3):
        wb = workloads.Workload(**{**w.__dict__, "seed": w.seed + 17 * b})
        inp = workloads.make_inputs(wb, "cuda")
        eo = None if w.identity_experts else workloads.make_expert_out(wb, max(wb.r_max, 1), "cuda")
        batches.append((wb, inp, eo))
    torch.cuda.synchronize()
    pipe = RoutePipeline(shape_of(w), "cuda")
    outs = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(9)]
    for i in range(9):  # every plan reused, batches in another cycle than the plans; no host sync
        wb, inp, eo = batches[i % 3]
        p = pipe.plan_for(pipe.step_index)
        pipe.step(inp["logits"], inp["x"], p.packed if eo is None else eo, inp["shared"], out=outs[i])
    assert pipe.status() == 0
    for i in range(9):
        wb, inp, eo = batches[i % 3]
        ref = RoutePlan(shape_of(w), "cuda")
        ref.step(inp["logits"], inp["x"], ref.packed if eo is None else eo, inp["shared"])
        assert ref.status() == 0
        y = bits(outs[i])
        assert np.array_equal(y, bits(ref.y[:w.T])), f"step {i}: y differs from the serial calls"
        if w.identity_experts:
            assert np.array_equal(y, bits(inp["x"])), "identity experts: combine(dispatch(x)) == x"


def test_pipeline_depth3_host_outputs():
    """Three plans, y and the statistics copied into pinned host buffers
    by the pipeline itself (the end-to-end path): y equals the serial calls
    bit for bit, aux and entropy are the oracle's (within 1e-9 and 1e-6)."""
    w = W["v2_top2"].scaled(1500)
    batches = []
    for b in range(4):
        wb = workloads.Workload(**{**w.__dict__, "seed": w.seed + 29 * b})
        eo = workloads.make_expert_out(wb, max(wb.r_max, 1), "cuda")
        batches.append((wb, workloads.make_inputs(wb, "cuda"), eo))
    pipe = RoutePipeline(shape_of(w), "cuda", depth=3)
    ys = [torch.empty((w.T, w.H), dtype=torch.bfloat16, pin_memory=True) for _ in range(8)]
    stats = [torch.empty(2, dtype=torch.float64, pin_memory=True) for _ in range(8)]
    for i in range(8):
        wb, inp, eo = batches[i % 4]
        pipe.step(inp["logits"], inp["x"], eo, inp["shared"], out=ys[i], stats_out=stats[i])
    assert pipe.status() == 0
    for i in range(8):
        wb, inp, eo = batches[i % 4]
        ref = RoutePlan(shape_of(w), "cuda")
        ref.step(inp["logits"], inp["x"], eo, inp["shared"])
        assert ref.status() == 0
        assert np.array_equal(bits(ys[i]), bits(ref.y[:w.T])), f"step {i}: y differs"
        og = oracle.gate(inp["logits"].cpu().numpy(), w.k, w.mode)
        assert abs(stats[i][0].item() - og[3]) <= 1e-9 and abs(stats[i][1].item() - og[4]) <= 1e-6


@pytest.mark.parametrize("depth,streams", [(2, 1), (3, 3)])
@pytest.mark.parametrize("w", [W["v2_top2"].scaled(1200), W["fp8_both"].scaled(700)], ids=lambda w: w.name)
def test_pipeline_plans_and_data_streams(w, depth, streams):
    """Other pipeline shapes: two plans with every data call on one stream,
    and three plans each with its own data stream (three batches' calls in
    flight at once) give the serial calls' bits."""
    batches = []
    for b in range(4):
        wb = workloads.Workload(**{**w.__dict__, "seed": w.seed + 13 * b})
        batches.append((workloads.make_inputs(wb, "cuda"), workloads.make_expert_out(wb, max(wb.r_max, 1), "cuda")))
    torch.cuda.synchronize()
    pipe = RoutePipeline(shape_of(w), "cuda", depth=depth, data_streams=streams)
    assert len(pipe.data_streams) == streams
    outs = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    for i in range(8):
        inp, eo = batches[i % 4]
        pipe.step(inp["logits"], inp["x"], eo, inp["shared"], out=outs[i])
    assert pipe.status() == 0
    for i in range(8):
        inp, eo = batches[i % 4]
        ref = RoutePlan(shape_of(w), "cuda")
        ref.step(inp["logits"], inp["x"], eo, inp["shared"])
        assert ref.status() == 0
        assert np.array_equal(bits(outs[i]), bits(ref.y[:w.T])), f"step {i}: y differs from the serial calls"
