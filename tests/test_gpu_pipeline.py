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
