"""The expert-parallel exchange on CPU ranks (gloo): every rank routes its
own batch (the oracle stands in for the kernels on CPU), sends each rank
its partition slice, applies that rank's experts, receives its rows back,
and combines.  The result must equal the same batch with every expert
local (no exchange), bit for bit, for world sizes 2 and 4, with and without
capacity drops, in bf16 and in FP8 (codes and scales travel together).

The de-duplicated exchange is checked the same way: each token goes to a
rank once with that rank's expert ids and gates, the receiver expands the
rows to its experts, combines each row's slots into one partial and sends
the partials back, and the source's sum of the partials equals the same
computation with every rank's experts local."""
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


def _rows_of(codes_or_bits, scales, oracle):
    """bf16 bits of the rows a receiver feeds its experts: the bf16 rows
    themselves, or e4m3 codes dequantised (zero + scale * value, fp32, one
    bf16 rounding) -- the expert's input transform, the same on both sides."""
    if scales is None:
        return codes_or_bits
    n, H = codes_or_bits.shape
    deq = np.array([[scales[r, 1] + scales[r, 0] * oracle.e4m3_decode(c) for c in codes_or_bits[r]]
                    for r in range(n)], dtype=np.float32).reshape(n, H)
    u = deq.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _expand_and_combine(oracle, rows_bits, slot_local, slot_gate, n_experts, expert0, k, H):
    """A receiver's work on de-duplicated rows: expand them to its experts
    (the layout of the rows' local slots, -1 = empty), run the experts, and
    combine each row's slots into one partial row (pinned fp32 order)."""
    n = slot_local.shape[0]
    if n == 0:
        return np.zeros((0, H), np.uint16), None
    Lr = oracle.layout(slot_local, n_experts, 1, 0, gates_f32=slot_gate)
    R = Lr["R"]
    packed = oracle.dispatch_bf16_rows(rows_bits, k, Lr["src_pos"], np.arange(R))
    eo = np.zeros((max(R, 1), H), np.uint16)
    for e in range(n_experts):
        r0, r1 = Lr["offsets"][e], Lr["offsets"][e + 1]
        eo[r0:r1] = _expert_fn(expert0 + e, packed[r0:r1])
    partials = oracle.combine_f32order(eo, Lr["gates"], Lr["dst_row"], np.arange(n), n, k)
    return partials, Lr


def _dedup_worker(rank, world, port, out_dir, cap_factor, fp8):
    """The de-duplicated exchange: send rows with one group per rank (a token
    goes to a rank once, with that rank's expert ids and gates), the receiver
    expands, runs its experts and returns one partial per row, the source adds
    the partials.  Compared with the same computation with every group
    local (no exchange)."""
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    from combine_moe_gate_warp_gb300 import workloads
    from combine_moe_gate_warp_gb300.ep import ExpertParallelExchange
    dist.init_process_group("gloo", rank=rank, world_size=world)
    base = workloads.Workload("epd", T=300, H=64, E=16, k=4, P=8, seed=910, capacity_factor=cap_factor)
    w = workloads.Workload(**{**base.__dict__, "seed": base.seed + 7919 * rank})
    T, H, E, k = w.T, w.H, w.E, w.k
    per = E // world
    logits = workloads.make_logits(w, "cpu").numpy()
    x = workloads.make_x(w, "cpu").view(torch.int16).numpy().view(np.uint16)
    idx, g64, *_ = oracle.gate(logits, k, w.mode)
    L = oracle.layout(idx, E, w.P, w.capacity, gates_f32=g64.astype(np.float32))
    Do = oracle.dedup_layout(L["dst_row"], L["offsets"], L["gates"], T, E, k, world)
    S = Do["S"]
    if fp8:
        send, scales = oracle.quantize_rows_grouped(x, Do["send_token"].astype(np.int64),
                                                    np.arange(S, dtype=np.int32), S)
        send_t, scales_t = torch.from_numpy(send), torch.from_numpy(scales)
    else:
        send = x[Do["send_token"]]
        scales = None
        send_t, scales_t = torch.from_numpy(send.view(np.int16)).view(torch.bfloat16), None
    ex = ExpertParallelExchange(E, w.P)
    rec = ex.dispatch_dedup(send_t, torch.from_numpy(Do["send_offsets"]), torch.from_numpy(Do["slot_local"]),
                            torch.from_numpy(Do["slot_gate"]), torch.from_numpy(L["counts"]), scales_t)
    # receiver: only this rank's experts arrive, each slot's count as announced
    ids = rec.slot_local.numpy()
    assert ids.shape == (rec.n, k) and np.all((ids >= -1) & (ids < per))
    rows_in = rec.rows.numpy() if fp8 else rec.rows.view(torch.int16).numpy().view(np.uint16)
    rows_bits = _rows_of(rows_in, None if rec.scales is None else rec.scales.numpy(), oracle)
    partials, Lr = _expand_and_combine(oracle, rows_bits, ids, rec.slot_gate.numpy(), per, rank * per, k, H)
    if Lr is not None:
        assert np.array_equal(Lr["counts"], rec.expert_counts.numpy())
    back = ex.combine_dedup(torch.from_numpy(partials.view(np.int16)).view(torch.bfloat16), rec, rows=S)
    back = back.view(torch.int16).numpy().view(np.uint16)[:S]
    y = oracle.combine_f32order(back if S else np.zeros((1, H), np.uint16), np.ones((T, world), np.float32),
                                Do["send_row"].ravel(), np.arange(T), T, world)
    # the same batch with every group local
    local = np.zeros((max(S, 1), H), np.uint16)
    src_bits = _rows_of(send, scales, oracle)
    for g in range(world):
        s0, s1 = int(Do["send_offsets"][g]), int(Do["send_offsets"][g + 1])
        part, _ = _expand_and_combine(oracle, src_bits[s0:s1], Do["slot_local"][s0:s1], Do["slot_gate"][s0:s1],
                                      per, g * per, k, H)
        local[s0:s1] = part
    y_ref = oracle.combine_f32order(local, np.ones((T, world), np.float32), Do["send_row"].ravel(), np.arange(T),
                                    T, world)
    np.savez(os.path.join(out_dir, f"d{rank}.npz"), y=y, y_ref=y_ref, back=back, local=local[:S], S=S, R=L["R"],
             n=rec.n, dropped=L["dropped"])
    dist.destroy_process_group()


@pytest.mark.parametrize("world,cap,fp8", [(2, 0.0, False), (4, 1.25, False), (4, 0.0, True), (2, 1.25, True)])
def test_dedup_exchange(tmp_path, oracle, world, cap, fp8):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_dedup_worker, args=(r, world, port, str(tmp_path), cap, fp8)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    res = [np.load(tmp_path / f"d{r}.npz") for r in range(world)]
    for r in res:
        assert np.array_equal(r["back"], r["local"]), "partials came back to the wrong send rows"
        assert np.array_equal(r["y"], r["y_ref"]), "combine of the exchanged partials differs"
        assert int(r["S"]) <= int(r["R"])  # a token goes to a rank at most once
    # every send row was received once, and fewer rows travel than packed rows
    assert sum(int(r["n"]) for r in res) == sum(int(r["S"]) for r in res)
    assert sum(int(r["S"]) for r in res) < sum(int(r["R"]) for r in res)
    if cap:
        assert any(int(r["dropped"]) > 0 for r in res)


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
