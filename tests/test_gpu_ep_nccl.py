"""The expert-parallel exchange over NCCL on the GPU with a world of one
rank (the only world this machine offers): the CUDA path routes and packs,
the exchange sends every partition to rank 0 and back through NCCL, and
moe_combine on the returned rows equals moe_combine on rows that never
left, bit for bit (bf16 and FP8 transport)."""
import socket

import numpy as np
import pytest
import torch

from combine_moe_gate_warp_gb300 import RoutePlan, workloads
from gpu_util import bits, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nccl_world():
    import torch.distributed as dist
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    yield
    dist.destroy_process_group()


def _expert(e, rows):
    return (rows.float() * ((e + 1) / 8.0)).to(torch.bfloat16)


@pytest.mark.parametrize("name", ["v2_top2", "fp8_skewed", "prefill_cap"])
def test_exchange_round_trip(nccl_world, name):
    from combine_moe_gate_warp_gb300.ep import ExpertParallelExchange
    w = workloads.WORKLOADS[name].scaled(2048)
    inp = workloads.make_inputs(w, "cuda")
    plan = RoutePlan(shape_of(w), "cuda")
    plan.gate(inp["logits"])
    plan.dispatch_layout()
    plan.dispatch(inp["x"])
    assert plan.status() == 0
    R = int(plan.layout.offsets[w.E].item())
    ex = ExpertParallelExchange(w.E, w.P)
    recv, recv_scales, recv_counts = ex.dispatch(plan.packed, plan.layout.counts, plan.scales)
    assert recv.shape[0] == R and torch.equal(recv, plan.packed[:R])
    if plan.scales is not None:
        assert torch.equal(recv_scales, plan.scales[:R])
        # the receiving side would dequantise; here the experts see the codes as values
        rows_in = recv.to(torch.bfloat16)
    else:
        rows_in = recv
    eo_recv = torch.empty((R, w.H), dtype=torch.bfloat16, device="cuda")
    for src, e, r0, r1 in ex.segments(recv_counts):
        eo_recv[r0:r1] = _expert(e, rows_in[r0:r1])
    eo_back = ex.combine(eo_recv, recv_counts, plan.layout.counts)
    plan.combine(eo_back, inp["shared"])
    y_ex = bits(plan.y[:w.T])
    eo_local = torch.empty_like(eo_recv)
    offs = plan.layout.offsets.cpu().tolist()
    for e in range(w.E):
        eo_local[offs[e]:offs[e + 1]] = _expert(e, rows_in[offs[e]:offs[e + 1]])
    plan.combine(eo_local, inp["shared"])
    assert plan.status() == 0
    assert np.array_equal(y_ex, bits(plan.y[:w.T]))
