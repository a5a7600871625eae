"""The expert-parallel exchange on CPU ranks (gloo): every rank routes its
own batch (the oracle stands in for the kernels on CPU), sends each rank
its partition slice, applies that rank's experts, receives its rows back,
and combines.  The result must equal the same batch with every expert
local (no exchange), bit for bit, for world sizes 2 and 4, with and without
capacity drops, in bf16 and in FP8 (codes and scales travel together)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _expert_fn(e, rows_bits):
    """A deterministic stand-in for expert e's FFN on bf16 rows: scale by
    (e + 1) / 8 in fp32, round to bf16 (round half to even)."""
    f = (rows_bits.astype(np.uint32) << 16).view(np.float32) * np.float32((e + 1) / 8.0)
    u = f.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _worker(rank, world, port, out_dir, cap_factor, fp8):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    from combine_moe_gate_warp_gb300 import workloads
    from combine_moe_gate_warp_gb300.ep import ExpertParallelExchange
    dist.init_process_group("gloo", rank=rank, world_size=world)
    base = workloads.Workload("ep", T=300, H=64, E=16, k=4, P=4, seed=900, capacity_factor=cap_factor)
    w = workloads.Workload(**{**base.__dict__, "seed": base.seed + 7919 * rank})
    logits = workloads.make_logits(w, "cpu").numpy()
    x = workloads.make_x(w, "cpu").view(torch.int16).numpy().view(np.uint16)
    idx, g64, *_ = oracle.gate(logits, w.k, w.mode)
    L = oracle.layout(idx, w.E, w.P, w.capacity, gates_f32=g64.astype(np.float32))
    R = L["R"]
    rows = np.arange(R, dtype=np.int64)
    ex = ExpertParallelExchange(w.E, w.P)
    counts = torch.from_numpy(L["counts"])
    if fp8:
        codes, scales = oracle.dispatch_fp8_rows(x, w.k, L["src_pos"], rows)
        recv, recv_scales, recv_counts = ex.dispatch(torch.from_numpy(codes), counts, torch.from_numpy(scales))
        # the receiving rank dequantises (zero + scale * value) and runs its experts
        recv_np = recv.numpy()
        sc = recv_scales.numpy()
        deq = np.array([[sc[r, 1] + sc[r, 0] * oracle.e4m3_decode(c) for c in recv_np[r]] for r in range(recv_np.shape[0])],
                       dtype=np.float32).reshape(recv_np.shape)
        recv_rows = (deq.view(np.uint32) + 0x7FFF + ((deq.view(np.uint32) >> 16) & 1)) >> 16
        recv_rows = recv_rows.astype(np.uint16)
    else:
        packed = oracle.dispatch_bf16_rows(x, w.k, L["src_pos"], rows)
        recv, _, recv_counts = ex.dispatch(torch.from_numpy(packed.view(np.int16)).view(torch.bfloat16), counts)
        recv_rows = recv.view(torch.int16).numpy().view(np.uint16)
    eo_recv = np.empty_like(recv_rows)
    for src, e, r0, r1 in ex.segments(recv_counts):
        assert e // (w.E // world) == rank  # only this rank's experts arrive here
        eo_recv[r0:r1] = _expert_fn(e, recv_rows[r0:r1])
    eo_back = ex.combine(torch.from_numpy(eo_recv.view(np.int16)).view(torch.bfloat16), recv_counts, counts)
    eo_back = eo_back.view(torch.int16).numpy().view(np.uint16)
    y = oracle.combine_f32order(eo_back if R else np.zeros((1, w.H), np.uint16), L["gates"], L["dst_row"],
                                np.arange(w.T), w.T, w.k)
    # the same batch with every expert local
    if fp8:
        deq_l = np.array([[scales[r, 1] + scales[r, 0] * oracle.e4m3_decode(c) for c in codes[r]] for r in range(R)],
                         dtype=np.float32).reshape(codes.shape)
        local_rows = ((deq_l.view(np.uint32) + 0x7FFF + ((deq_l.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    else:
        local_rows = packed
    eo_local = np.empty_like(local_rows)
    for e in range(w.E):
        r0, r1 = L["offsets"][e], L["offsets"][e + 1]
        eo_local[r0:r1] = _expert_fn(e, local_rows[r0:r1])
    y_ref = oracle.combine_f32order(eo_local if R else np.zeros((1, w.H), np.uint16), L["gates"], L["dst_row"],
                                    np.arange(w.T), w.T, w.k)
    np.savez(os.path.join(out_dir, f"r{rank}.npz"), y=y, y_ref=y_ref, eo_back=eo_back, eo_local=eo_local,
             recv_counts=recv_counts.numpy(), R=R, dropped=L["dropped"])
    dist.destroy_process_group()


@pytest.mark.parametrize("world,cap,fp8", [(2, 0.0, False), (4, 1.25, False), (2, 1.25, True)])
def test_expert_parallel_exchange(tmp_path, oracle, world, cap, fp8):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, str(tmp_path), cap, fp8)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    res = [np.load(tmp_path / f"r{r}.npz") for r in range(world)]
    for r in res:
        assert np.array_equal(r["eo_back"], r["eo_local"]), "rows came back to the wrong places"
        assert np.array_equal(r["y"], r["y_ref"]), "combine after the exchange differs"
    # every row a rank sent was received by someone: totals match
    assert sum(int(r["recv_counts"].sum()) for r in res) == sum(int(r["R"]) for r in res)


def _short_worker(rank, world, port, out_dir):
    """Rank 1 hands the exchange a packed buffer shorter than its counts: it
    must refuse before any collective, and rank 0's exchange must end with
    an error (the process group's short timeout), not hang."""
    import datetime
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from combine_moe_gate_warp_gb300.ep import ExpertParallelExchange
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
    ex = ExpertParallelExchange(8, 2)
    counts = torch.tensor([3, 1, 2, 2, 0, 4, 1, 1], dtype=torch.int32)
    packed = torch.zeros((14 if rank == 0 else 9, 16), dtype=torch.bfloat16)
    err = "none"
    try:
        ex.dispatch(packed, counts)
    except ValueError as e:
        err = "refused: " + str(e)
    except Exception as e:  # the peer's collective ends with the group's timeout
        err = "failed: " + type(e).__name__
    with open(os.path.join(out_dir, f"s{rank}.txt"), "w") as f:
        f.write(err)
    os._exit(0)


def test_short_send_is_refused_and_the_peer_fails(tmp_path):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_short_worker, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    r0 = (tmp_path / "s0.txt").read_text()
    r1 = (tmp_path / "s1.txt").read_text()
    assert r1.startswith("refused"), r1
    assert r0.startswith("failed"), r0
