"""The expert-parallel exchange over NCCL on the GPU with a world of one
rank (the only world this machine offers): the CUDA path routes and packs,
the exchange sends every partition to rank 0 and back through NCCL, and
moe_combine on the returned rows equals moe_combine on rows that never
left, bit for bit (bf16 and FP8 transport).  The de-duplicated form sends
each token once with its expert ids and gates, the receiver expands and
combines them with the library calls, and moe_combine_partials on the
returned partial rows equals the same calls without the exchange."""
import socket

import numpy as np
import pytest
import torch

from combine_moe_gate_warp_gb300 import RoutePlan, RouteShape, abi, workloads
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
    eo_back = ex.combine(eo_recv, recv_counts, plan.layout)  # r_max rows, as moe_combine requires
    assert eo_back.shape[0] == max(plan.r_max, 1)
    plan.combine(eo_back, inp["shared"])
    y_ex = bits(plan.y[:w.T])
    eo_local = torch.empty_like(eo_back)
    offs = plan.layout.offsets.cpu().tolist()
    for e in range(w.E):
        eo_local[offs[e]:offs[e + 1]] = _expert(e, rows_in[offs[e]:offs[e + 1]])
    plan.combine(eo_local, inp["shared"])
    assert plan.status() == 0
    assert np.array_equal(y_ex, bits(plan.y[:w.T]))


def _expand_and_combine(rows, slot_local, slot_gate, expert_counts, E, k, H):
    """A receiver's calls on de-duplicated rows: the layout of their slots
    (-1 = empty), the copies to its experts, the experts, and the combine of
    each row's slots into one partial row.  Returns the partials [n, H]."""
    n = rows.shape[0]
    rp = RoutePlan(RouteShape(T=n, H=H, E=E, k=k, P=1), "cuda")
    rp.topk_idx[:n].copy_(slot_local)
    rp.gates[:n].copy_(slot_gate)
    rp.expert_counts.copy_(expert_counts)
    rp.dispatch_layout()
    rp.dispatch(rows[:n])
    eo = torch.empty((max(rp.r_max, 1), H), dtype=torch.bfloat16, device="cuda")
    offs = rp.layout.offsets.cpu().tolist()
    for e in range(E):
        eo[offs[e]:offs[e + 1]] = _expert(e, rp.packed[offs[e]:offs[e + 1]])
    rp.combine(eo)
    assert rp.status() == 0
    return rp.y[:n].clone()


@pytest.mark.parametrize("name", ["v2_top2", "fine_shared", "prefill_cap", "prefill_reassign"])
def test_dedup_exchange_round_trip(nccl_world, name):
    from combine_moe_gate_warp_gb300.ep import ExpertParallelExchange
    w = workloads.WORKLOADS[name].scaled(2048)
    T, H, E, k = w.T, w.H, w.E, w.k
    inp = workloads.make_inputs(w, "cuda")
    plan = RoutePlan(shape_of(w), "cuda")
    plan.gate(inp["logits"])
    plan.dispatch_layout()
    assert plan.status() == 0
    ex = ExpertParallelExchange(E, w.P)
    D = abi.Dedup(T, k, ex.W, "cuda")
    abi.moe_dedup_layout(plan.layout, plan.gates, D, groups=ex.W)  # one group per rank
    send = torch.empty((D.s_max, H), dtype=torch.bfloat16, device="cuda")
    abi.moe_dispatch_dedup(inp["x"], T, H, D, 0, send)
    rec = ex.dispatch_dedup(send, D.send_offsets, D.slot_local, D.slot_gate, plan.layout)
    S = int(D.send_offsets[ex.W].item())
    assert rec.n == S and torch.equal(rec.rows, send[:S])
    assert torch.equal(rec.expert_counts, plan.layout.counts)
    partials = _expand_and_combine(rec.rows, rec.slot_local, rec.slot_gate, rec.expert_counts, E, k, H)
    back = ex.combine_dedup(partials, rec, rows=D.s_max)
    assert back.shape[0] == D.s_max
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    abi.moe_combine_partials(back, D, inp["shared"], w.Ks, T, H, y)
    # the same calls on the send rows that never left
    local = _expand_and_combine(send[:S], D.slot_local[:S], D.slot_gate[:S], plan.layout.counts, E, k, H)
    back_l = torch.empty((D.s_max, H), dtype=torch.bfloat16, device="cuda")
    back_l[:S] = local
    y_l = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    abi.moe_combine_partials(back_l, D, inp["shared"], w.Ks, T, H, y_l)
    assert plan.status() == 0
    assert np.array_equal(bits(back[:S]), bits(local))
    assert np.array_equal(bits(y), bits(y_l))
    if not w.Ks:
        # one rank: a token's partial is its whole routed sum, so y equals the plain path's
        plan.dispatch(inp["x"])
        eo = torch.empty((max(plan.r_max, 1), H), dtype=torch.bfloat16, device="cuda")
        offs = plan.layout.offsets.cpu().tolist()
        for e in range(E):
            eo[offs[e]:offs[e + 1]] = _expert(e, plan.packed[offs[e]:offs[e + 1]])
        plan.combine(eo)
        assert plan.status() == 0
        assert np.array_equal(bits(y), bits(plan.y[:T]))


def test_dedup_exchange_fp8_bytes(nccl_world):
    """FP8 send rows: codes, scales, ids and gates arrive unchanged."""
    from combine_moe_gate_warp_gb300.ep import ExpertParallelExchange
    w = workloads.WORKLOADS["fp8_skewed"].scaled(3000)
    T, H, E, k = w.T, w.H, w.E, w.k
    inp = workloads.make_inputs(w, "cuda")
    plan = RoutePlan(shape_of(w), "cuda")
    plan.gate(inp["logits"])
    plan.dispatch_layout()
    ex = ExpertParallelExchange(E, w.P)
    D = abi.Dedup(T, k, ex.W, "cuda")
    abi.moe_dedup_layout(plan.layout, plan.gates, D, groups=ex.W)
    send = torch.empty((D.s_max, H), dtype=torch.uint8, device="cuda")
    sc = torch.empty((D.s_max, 2), dtype=torch.float32, device="cuda")
    abi.moe_dispatch_dedup(inp["x"], T, H, D, 1, send, sc)
    rec = ex.dispatch_dedup(send, D.send_offsets, D.slot_local, D.slot_gate, plan.layout, sc)
    assert plan.status() == 0
    S = rec.n
    assert torch.equal(rec.rows, send[:S]) and torch.equal(rec.scales, sc[:S])
    assert torch.equal(rec.slot_local, D.slot_local[:S]) and torch.equal(rec.slot_gate, D.slot_gate[:S])
