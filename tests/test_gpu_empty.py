"""Empty batches (T = 0) through every entry point added beyond the four
forward calls: nothing is written beyond the zero-sized outputs, the
summary arrays are zero, and the device status stays clean."""
import pytest
import torch

from combine_moe_gate_warp_gb300 import RoutePlan, abi, workloads
from gpu_util import shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    torch.cuda.init()


@pytest.mark.parametrize("fp8,fp8c,reassign", [(2, 0, False), (3, 1, False), (1, 2, True), (0, 3, True)])
def test_empty_batch_everywhere(fp8, fp8c, reassign):
    w = workloads.Workload("empty", T=0, H=64, E=16, k=4, P=4, fp8=fp8, fp8_combine=fp8c,
                           capacity_factor=1.25 if reassign else 0.0, reassign=reassign, seed=5)
    plan = RoutePlan(shape_of(w), "cuda")
    inp = workloads.make_inputs(w, "cuda")
    plan.step(inp["logits"], inp["x"], workloads.make_expert_out(w, 1, "cuda"), inp["shared"])
    assert plan.status() == 0
    assert plan.layout.offsets.cpu().tolist() == [0] * 17
    assert plan.layout.part_tokens.cpu().tolist() == [0] * 4
    D = abi.Dedup(0, w.k, w.P, "cuda")
    abi.moe_dedup_layout(plan.layout, plan.gates, D)
    send = torch.empty((1, w.H), dtype=torch.bfloat16, device="cuda")
    abi.moe_dispatch_dedup(inp["x"], 0, w.H, D, 0, send)
    y = torch.empty((1, w.H), dtype=torch.bfloat16, device="cuda")
    abi.moe_combine_partials(send, D, None, 0, 0, w.H, y)
    assert plan.status() == 0
    assert D.send_offsets.cpu().tolist() == [0] * 5
    dy = torch.empty((0, w.H), dtype=torch.bfloat16, device="cuda")
    plan.combine_backward(dy, workloads.make_expert_out(w, 1, "cuda"))
    plan.gate_backward(inp["logits"], torch.empty((0, w.k), dtype=torch.float32, device="cuda"))
    plan.dispatch_backward(workloads.make_expert_out(w, 1, "cuda"))
    assert plan.status() == 0
