"""Error paths on the GPU: host argument checks leave nothing enqueued;
device-detected problems land in the workspace status word; a look-back
wait that nothing satisfies expires after its bound and reports
MOE_ERR_TIMEOUT instead of hanging.  No test faults or traps the GPU: every
failure is made on the host (bad arguments, corrupted inputs, a workspace
hook that makes one tile skip publishing)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import RoutePlan, RouteShape, abi, workloads
from gpu_util import route_checked, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()


def _plan(T=600, E=16, k=2, P=4, H=64, cap=0):
    return RoutePlan(RouteShape(T=T, H=H, E=E, k=k, P=P, capacity=cap), "cuda")


def test_host_argument_errors():
    p = _plan()
    logits = torch.randn(600, 16, device="cuda")
    with pytest.raises(abi.MoeError) as e:
        abi.moe_gate(logits, 0, 0, p.topk_idx, p.gates, p.expert_counts, p.aux_loss, p.entropy, p.ws)
    assert e.value.status == abi.MOE_ERR_UNSUPPORTED
    with pytest.raises(abi.MoeError) as e:
        abi.moe_gate(logits, 2, 7, p.topk_idx, p.gates, p.expert_counts, p.aux_loss, p.entropy, p.ws)
    assert e.value.status == abi.MOE_ERR_INVALID_ARG
    big = torch.randn(601 * 16 + 1, device="cuda")[1:].view(601, 16)  # 4-byte misaligned base
    with pytest.raises(abi.MoeError) as e:
        abi.moe_gate(big, 2, 0, p.topk_idx, p.gates, p.expert_counts, p.aux_loss, p.entropy, p.ws)
    assert e.value.status == abi.MOE_ERR_INVALID_ARG
    small_ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(abi.MoeError) as e:
        abi.moe_dispatch_layout(p.topk_idx, p.expert_counts, 600, 16, 2, 4, 0, None, p.layout, small_ws)
    assert e.value.status == abi.MOE_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(abi.MoeError) as e:  # P does not divide E
        abi.moe_dispatch_layout(p.topk_idx, p.expert_counts, 600, 16, 2, 3, 0, None, p.layout, p.ws)
    assert e.value.status == abi.MOE_ERR_UNSUPPORTED
    x = torch.randn(600, 64, device="cuda").bfloat16()
    p.gate(logits)
    p.dispatch_layout()
    with pytest.raises(abi.MoeError) as e:  # H not a multiple of 16 for FP8
        abi.moe_dispatch(x[:, :40].contiguous(), 600, 40, p.layout, 1,
                         torch.empty(p.r_max, 40, dtype=torch.uint8, device="cuda"),
                         torch.empty(p.r_max, 2, device="cuda"))
    assert e.value.status == abi.MOE_ERR_UNSUPPORTED
    with pytest.raises(abi.MoeError) as e:  # T disagrees with the layout
        abi.moe_dispatch(x, 599, 64, p.layout, 0, p.packed)
    assert e.value.status == abi.MOE_ERR_INVALID_ARG
    assert p.status() == 0  # nothing above reached the device


def test_non_finite_logits_reported():
    p = _plan()
    logits = torch.randn(600, 16, device="cuda")
    logits[17, 3] = float("nan")
    logits[400, 0] = float("inf")
    p.gate(logits)
    assert p.status() == abi.MOE_ERR_DEVICE_DATA
    p.gate(torch.randn(600, 16, device="cuda"))
    assert p.status() == 0  # cleared by the read, and the workspace is clean


def test_out_of_range_ids_and_count_mismatch_reported():
    w = workloads.Workload("bad", T=600, H=64, E=16, k=2, P=4, seed=11)
    p = RoutePlan(shape_of(w), "cuda")
    inp = workloads.make_inputs(w, "cuda")
    p.gate(inp["logits"])
    assert p.status() == 0
    p.topk_idx[5, 1] = 16
    p.topk_idx[300, 0] = -3
    p.dispatch_layout()
    assert p.status() == abi.MOE_ERR_DEVICE_DATA
    d = p.layout.dst_row.cpu().numpy()
    assert d[11] == -1 and d[600] == -1       # the bad slots are dropped
    R = int(p.layout.offsets[16].item())
    assert R <= p.r_max and np.all(d < p.r_max)
    # counts that do not match the ids
    p.gate(inp["logits"])
    p.expert_counts[0] += 5
    p.dispatch_layout()
    assert p.status() == abi.MOE_ERR_DEVICE_DATA
    # a clean call afterwards is exact again
    route_checked(w, p, inp["logits"])


def test_lookback_wait_expires_with_timeout_status():
    """Tile 1 of the layout is told (through the workspace hook, from the
    host) not to publish; tile 2's bounded wait expires after ~1 s and the
    call reports MOE_ERR_TIMEOUT.  The context stays usable."""
    w = workloads.Workload("timeout", T=4 * 512, H=64, E=16, k=2, P=4, seed=12)
    p = RoutePlan(shape_of(w), "cuda")
    inp = workloads.make_inputs(w, "cuda")
    p.gate(inp["logits"])
    assert p.status() == 0
    p.ws.view(torch.int32)[3] = 2  # inject_skip_publish (byte offset 12) = tile 1 + 1
    p.dispatch_layout()
    assert p.status() == abi.MOE_ERR_TIMEOUT
    # the hook is cleared and the workspace usable again
    route_checked(w, p, inp["logits"])


def test_route_non_finite_logits_reported():
    p = _plan()
    assert p.fused_route
    logits = torch.randn(600, 16, device="cuda")
    logits[17, 3] = float("nan")
    logits[400, 0] = float("inf")
    p.route(logits)
    assert p.status() == abi.MOE_ERR_DEVICE_DATA
    p.route(torch.randn(600, 16, device="cuda"))
    assert p.status() == 0


def test_route_wait_expires_with_timeout_status():
    """moe_route: tile 1 is told (through the workspace hook, from the host)
    never to arrive at the grid-wide wait; the other tiles' bounded wait
    expires after ~1 s and the call reports MOE_ERR_TIMEOUT.  Reading the
    status re-arms the workspace: the next calls (both parities of the
    barrier) are exact again."""
    w = workloads.Workload("timeout_route", T=4096, H=64, E=16, k=2, P=4, seed=13)
    p = RoutePlan(shape_of(w), "cuda")
    assert p.fused_route
    inp = workloads.make_inputs(w, "cuda")
    route_checked(w, p, inp["logits"])
    p.ws.view(torch.int32)[3] = 2  # inject_skip_publish (byte offset 12) = tile 1 + 1
    p.route(inp["logits"])
    assert p.status() == abi.MOE_ERR_TIMEOUT
    assert int(p.ws.view(torch.int32)[3].item()) == 0  # the hook was consumed
    for _ in range(3):
        route_checked(w, p, inp["logits"])


def test_route_launches_query():
    """moe_route_launches: 1 (the fused kernel) for the batches used here, 2
    (gate and layout kernels) for a batch whose tiles cannot fit in shared
    memory, 0 for unsupported sizes; the plan counts its launches with it.
    Only the occupancy of the kernel is queried: nothing is launched."""
    for name in ("tiny", "v2_top2", "fine_shared", "fp8_skewed", "prefill_cap"):
        w = workloads.WORKLOADS[name]
        assert abi.moe_route_launches(w.T, w.E, w.k, w.mode, w.P) == 1, name
    assert abi.moe_route_launches(1 << 25, 256, 16, 0, 8) == 2
    assert abi.moe_route_launches(100, 8, 9, 0, 4) == 0   # k > E for the gate
    assert abi.moe_route_launches(100, 8, 2, 5, 4) == 0   # bad mode
    p = _plan()
    assert p.launches_per_step() == 3
