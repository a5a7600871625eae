"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2):
barrier + MAX all-reduce of the timing, per-rank independent batches, and
the data-parallel property that makes the path shard without an exchange
(routing each rank's tokens alone equals routing them as one batch, for the
token-parallel gate; each rank's layout only indexes its own tokens)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import oracle
    from combine_moe_gate_warp_gb300 import workloads
    bench.init_dist(world, "gloo")
    base = workloads.WORKLOADS["tiny"]
    w = bench.rank_workload(base, rank)
    logits = workloads.make_logits(w, "cpu").numpy()
    idx, g, counts, aux, ent = oracle.gate(logits, w.k, w.mode)
    L = oracle.layout(idx, w.E, w.P, 0)
    bench.barrier(world)
    t = bench.max_over_ranks(1.5 + rank, world)
    np.savez(os.path.join(out_dir, f"r{rank}.npz"), logits=logits, idx=idx, g=g, counts=counts,
             src_pos=L["src_pos"], t=t, seed=w.seed)
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path, oracle):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    r = [np.load(tmp_path / f"r{i}.npz") for i in range(2)]
    assert r[0]["t"] == r[1]["t"] == 2.5            # MAX over ranks
    assert r[0]["seed"] != r[1]["seed"]             # own batch per rank
    assert not np.array_equal(r[0]["logits"], r[1]["logits"])
    # token-parallel gate: the concatenated batch routes like its shards
    both = np.concatenate([r[0]["logits"], r[1]["logits"]])
    idx, g, counts, _, _ = oracle.gate(both, 2, 0)
    assert np.array_equal(idx, np.concatenate([r[0]["idx"], r[1]["idx"]]))
    assert np.array_equal(g, np.concatenate([r[0]["g"], r[1]["g"]]))
    assert np.array_equal(counts, r[0]["counts"] + r[1]["counts"])
    # each rank's packed rows come from its own tokens only
    for i in range(2):
        assert r[i]["src_pos"].max() < 256 * 2
