#!/usr/bin/env python3
"""Benchmark of the MoE token-routing hot path on GB300.

One step = moe_gate -> moe_dispatch_layout -> moe_dispatch -> moe_combine
over one batch of synthetic, seeded input already resident in HBM (expert
outputs are seeded inputs: the expert FFN is not part of this path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle, as the reference arm)

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank routes its
own batch (data parallel, no collective on the data path: weak scaling); the
timed region is bracketed by a barrier and a device synchronise and the
slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "route+dispatch+combine tokens/s and HBM GB/s (fraction of GB300 roofline)"
UNIT = "tokens/s"
# the workloads a default run times; the line's headline is the largest
DEFAULT_WORKLOADS = ("v2_top2", "fine_shared", "fp8_skewed", "prefill_cap")
HEADLINE_WORKLOAD = "prefill_cap"  # batch 128 x seq 2048, hidden 4096, 64 experts, top-8, capacity 1.25


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", "--config", default="all",
                    help="'all' (v2_top2, fine_shared, fp8_skewed and prefill_cap in one run, the headline on "
                         "prefill_cap), a workload name, or C0..C4 for tiny, v2_top2, fine_shared, fp8_skewed, "
                         "prefill_cap")
    ap.add_argument("--seed", type=int, default=None, help="override the workload's seed")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (a smaller case of the same shape, e.g. to profile)")
    ap.add_argument("--oracle-threads", type=int, default=0,
                    help="threads of the second oracle baseline (0: every core this process may use)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample of the headline workload")
    ap.add_argument("--cpu-seconds-other", type=float, default=3.0,
                    help="target CPU time of the oracle baseline sample of each other workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-pipeline", action="store_true",
                    help="do not time the back-to-back batches of RoutePipeline")
    ap.add_argument("--no-graph", action="store_true",
                    help="do not time the step captured as a CUDA graph (RouteGraph)")
    ap.add_argument("--data-streams", type=int, choices=[0, 1, 2], default=0,
                    help="streams the pipelined batches' dispatch and combine alternate over, with two "
                         "plans (0: time the configurations of PIPE_CONFIGS and keep the fastest)")
    ap.add_argument("--route-priority", choices=["high", "same"], default="high",
                    help="priority of the routing stream against the data stream")
    ap.add_argument("--dedup-steps", type=int, default=200,
                    help="passes of the per-partition de-duplicated send path timed after the forward (0: skip)")
    ap.add_argument("--backward-steps", type=int, default=500,
                    help="passes of the backward calls timed after the forward (0: skip)")
    args = ap.parse_args()
    aliases = {"C0": "tiny", "C1": "v2_top2", "C2": "fine_shared", "C3": "fp8_skewed", "C4": "prefill_cap"}
    args.workload = aliases.get(args.workload, args.workload)
    return args


def resolve_workload(args):
    """The named workload with the --seed and --tokens overrides applied."""
    from combine_moe_gate_warp_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    if args.seed is not None:
        w = workloads.Workload(**{**w.__dict__, "seed": args.seed})
    if args.tokens is not None:
        w = w.scaled(args.tokens)
    return w


# ---------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks only)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region (nvidia-smi sampler)
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, bus_id: str | None, period_ms: int = 100):
        self.samples = []  # (host time, dict)
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            bus = parts[0].lower()
            if self.bus_id and not (bus.endswith(self.bus_id[-12:]) or self.bus_id.endswith(bus[-12:])):
                continue
            try:
                d = dict(sm=float(parts[1]), sm_max=float(parts[2]),
                         power=float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None,
                         active=parts[4], hw_slowdown=parts[5], hw_thermal=parts[6],
                         sw_thermal=parts[7], sw_power_cap=parts[8])
            except ValueError:
                continue
            self.samples.append((time.time(), d))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [d for (t, d) in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside and self.samples:
            # nearest samples when the timed region is shorter than the period
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
            note = "nearest sample to the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        reasons = set()
        for d in inside:
            for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
                if d[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(d["sm"] for d in inside),
                "sm_max_mhz": max(d["sm_max"] for d in inside),
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# byte accounting of the roofline (algorithmic bytes, not measured traffic)
# ---------------------------------------------------------------------------
def kernel_bytes(w, R):
    """Algorithmic bytes per call of the step (and of the whole step)."""
    bt = 1 if w.fp8 else 2
    x = w.T * w.H * 2
    grouped = int(w.fp8) in (2, 3)
    # grouped FP8 modes read x once more for the group extremes
    packed = R * w.H * bt + (R * 8 if w.fp8 else 0)
    y = w.T * w.H * 2
    shared = w.Ks * w.T * w.H * 2
    by = {
        "gate": w.T * w.E * 4 + w.T * w.k * 8 + w.E * 4,
        "layout": w.T * w.k * (4 + 4 + 1 + 4) + R * 4,
        "dispatch": x * (2 if grouped else 1) + packed,
    }
    # the fused routing call: logits read, ids, gates, dst_row, mask and src_pos written
    by["route"] = w.T * w.E * 4 + w.T * w.k * (4 + 4 + 4 + 1) + R * 4
    if w.fp8_combine:
        # expert side: bf16 rows read (twice for grouped modes), codes and scales written;
        # combine: codes and scales read
        qgrouped = int(w.fp8_combine) in (2, 3)
        by["quantize"] = R * w.H * 2 * (2 if qgrouped else 1) + R * (w.H + 8)
        by["combine"] = R * (w.H + 8) + y + shared + w.T * w.k * 8
        eo_metric = R * w.H * 2 + R * w.H + R * w.H  # bf16 read, codes written, codes read
    else:
        by["combine"] = R * w.H * 2 + y + shared + w.T * w.k * 8
        eo_metric = R * w.H * 2
    # the metric's bytes: x read, packed written, expert outputs read (for FP8
    # expert outputs: read in bf16, codes written and read), y written
    by["roofline_step"] = x + R * w.H * bt + eo_metric + y
    # every byte the step moves
    by["all_step"] = sum(v for k2, v in by.items() if k2 not in ("roofline_step", "gate", "layout"))
    return by


def kernel_sources(name: str, w=None) -> tuple:
    """Source files of the kernel behind a call (for the traffic table's
    staleness check)."""
    fp8 = bool(w is not None and w.fp8)
    fp8c = bool(w is not None and w.fp8_combine)
    table = {
        "gate": ("gate.cu",), "layout": ("layout.cu",), "route": ("route.cu", "tma.cuh"),
        "dispatch": ("quant.cu", "fp8.cuh", "tma.cuh") if fp8 else ("dispatch.cu", "tma.cuh"),
        "quantize": ("quant.cu", "fp8.cuh", "tma.cuh"),
        "combine": ("quant.cu", "fp8.cuh") if fp8c else ("combine.cu", "tma.cuh"),
        "combine_backward": ("backward.cu",), "gate_backward": ("backward.cu",),
        "dispatch_backward": ("combine.cu", "tma.cuh"),
    }
    return table[name] + ("common.cuh",)


def source_digest(name: str, w=None) -> str:
    csrc = os.path.join(ROOT, "combine_moe_gate_warp_gb300", "csrc")
    h = hashlib.sha256()
    for f in kernel_sources(name, w):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str, w=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(workload, {}).get(kernel)
    if not ent or ent.get("source_digest") != source_digest(kernel, w):
        return None
    return ent.get("dram_bytes_per_launch")


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------
def _ranges(n, parts):
    """Split [0, n) into `parts` contiguous ranges (as int64 index arrays)."""
    import numpy as np
    edges = np.linspace(0, n, parts + 1).astype(np.int64)
    return [np.arange(edges[i], edges[i + 1], dtype=np.int64) for i in range(parts) if edges[i + 1] > edges[i]]


def oracle_sample_run(w, inputs_host, T_s, threads=1):
    """Time the oracle on the first T_s tokens of the workload: gate, layout,
    dispatch of every kept row, combine of every token.  Returns seconds.
    With threads > 1 the per-token and per-row stages (gate, dispatch,
    combine, the FP8 encodes) run over contiguous token / row ranges on a
    thread pool (the C oracle releases the interpreter lock); the layout's
    sort and the FP8 group extremes stay serial."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    logits = inputs_host["logits"][:T_s]
    x_bits = inputs_host["x"][:T_s]
    cap = 0
    if w.capacity:
        cap = (5 * T_s * w.k + 4 * w.E - 1) // (4 * w.E)
    pool = cf.ThreadPoolExecutor(max_workers=threads) if threads > 1 else None

    def pmap(fn, parts):
        return list(pool.map(fn, parts)) if pool else [fn(q) for q in parts]

    def quantize(src, src_row, mode, offsets, rows):
        group, ng = oracle.row_groups(mode, offsets, rows)
        if mode == oracle.FP8_PER_TOKEN:
            parts = pmap(lambda r: oracle.quantize_rows_grouped(src, src_row[r], np.arange(r.size, dtype=np.int32),
                                                                r.size), _ranges(rows.size, threads))
        else:
            params = oracle.fp8_group_params(src, src_row, group, ng)
            parts = pmap(lambda r: oracle.quantize_rows_with_params(src, src_row[r], group[r], params),
                         _ranges(rows.size, threads))
        if not parts:
            return np.zeros((0, src.shape[1]), np.uint8), np.zeros((0, 2), np.float32)
        return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])

    t0 = time.perf_counter()
    gparts = pmap(lambda r: oracle.gate(logits[r[0]:r[-1] + 1], w.k, w.mode), _ranges(T_s, threads))
    idx = np.concatenate([g[0] for g in gparts])
    g64 = np.concatenate([g[1] for g in gparts])
    if w.reassign and cap:
        L = oracle.layout_reassign(idx, w.E, w.P, cap, gates_f32=g64.astype(np.float32))
    else:
        L = oracle.layout(idx, w.E, w.P, cap, gates_f32=g64.astype(np.float32))
    rows = np.arange(L["R"], dtype=np.int64)
    src_row = L["src_pos"].astype(np.int64) // w.k
    if w.fp8:
        packed, scales = quantize(x_bits, src_row, int(w.fp8), L["offsets"], rows)
    else:
        packed = np.concatenate(pmap(lambda r: oracle.dispatch_bf16_rows(x_bits, w.k, L["src_pos"], r),
                                     _ranges(L["R"], threads)) or [np.zeros((0, w.H), np.uint16)])
    t1 = time.perf_counter()
    eo = packed if w.identity_experts else inputs_host["eo"][:max(L["R"], 1)]
    sh = None if inputs_host.get("shared") is None else np.ascontiguousarray(inputs_host["shared"][:, :T_s])
    t2 = time.perf_counter()
    if w.fp8_combine:
        codes, sc = quantize(eo, rows, int(w.fp8_combine), L["offsets"], rows)
        pmap(lambda r: oracle.combine_fp8_f32order(codes, sc, L["gates"], L["dst_row"], r, T_s, w.k, sh),
             _ranges(T_s, threads))
    else:
        pmap(lambda r: oracle.combine_f32order(eo, L["gates"], L["dst_row"], r, T_s, w.k, sh), _ranges(T_s, threads))
    t3 = time.perf_counter()
    if pool:
        pool.shutdown()
    return (t1 - t0) + (t3 - t2)


def host_cpu():
    """(usable cores, CPU model) of this host."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
        for key in ("model name", "CPU part"):
            hit = [ln.split(":", 1)[1].strip() for ln in info if ln.startswith(key)]
            if hit:
                model = hit[0] if key == "model name" else f"Arm CPU part {hit[0]}"
                break
    except OSError:
        pass
    return cores, model or "unknown"


HOST_EO_ROWS = 1 << 17  # cap on host copies of the seeded expert outputs


def max_sample_tokens(w):
    return w.T if w.identity_experts else min(w.T, HOST_EO_ROWS // w.k)


def cpu_baseline(w, inputs_host, target_s, threads=0):
    """Scale the token sample so that one oracle pass takes about target_s
    seconds (whole workload at most), then time it."""
    T_max = max_sample_tokens(w)
    T_s = min(T_max, 256)
    dt = oracle_sample_run(w, inputs_host, T_s)
    while dt < 0.25 * target_s and T_s < T_max:
        T_s = min(T_max, max(T_s * 2, int(T_s * target_s / max(dt, 1e-6) * 0.8)))
        dt = oracle_sample_run(w, inputs_host, T_s)
    reps = 1
    total = dt
    while total < 0.5 * target_s and reps < 50:
        total += oracle_sample_run(w, inputs_host, T_s)
        reps += 1
    single = dict(value=T_s * reps / total, unit=UNIT, cores=1, kind="oracle",
                  sample=f"first {T_s} of {w.T} tokens of {w.name}, whole path (gate, layout, "
                         f"dispatch of every kept row, combine of every token), {reps} pass(es), "
                         f"{total:.1f} s single-threaded C oracle")
    cores, model = host_cpu()
    if threads > 0:
        cores = threads
    if cores > 1:
        tm = sum(oracle_sample_run(w, inputs_host, T_s, cores) for _ in range(reps))
        single["threaded"] = dict(value=T_s * reps / tm, unit=UNIT, cores=cores, cpu=model,
                                  sample=f"the same sample, {reps} pass(es), per-token and per-row stages over "
                                         f"{cores} threads (token / row ranges), layout sort serial")
    single["cpu"] = model
    return single


def host_inputs(w, inputs, eo):
    import numpy as np
    import torch
    d = dict(logits=inputs["logits"].cpu().numpy(),
             x=inputs["x"].cpu().view(torch.int16).numpy().view(np.uint16))
    if eo is not None:
        d["eo"] = eo[:HOST_EO_ROWS].cpu().view(torch.int16).numpy().view(np.uint16)
    if inputs.get("shared") is not None:
        d["shared"] = inputs["shared"].cpu().view(torch.int16).numpy().view(np.uint16)
    return d


def rank_workload(base, rank: int):
    """Data-parallel sharding: every rank routes its own batch of the same
    shape (its own seed); nothing on the data path is exchanged."""
    from combine_moe_gate_warp_gb300 import workloads
    return workloads.Workload(**{**base.__dict__, "seed": base.seed + 7919 * rank})


def config_of(w, world):
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "P": w.P,
            "gate": "softmax_topk" if w.mode else "topk_softmax",
            "transport": (["bf16", "e4m3 per-token", "e4m3 per-expert", "e4m3 global"][int(w.fp8)]),
            "expert_outputs": (["bf16", "e4m3 per-token", "e4m3 per-expert", "e4m3 global"][int(w.fp8_combine)]),
            "Ks": w.Ks,
            "capacity": w.capacity or None,
            "overflow": ("re-assigned to the least-loaded expert" if w.reassign else "dropped") if w.capacity else None,
            "l2": "no flush: each step touches ~%.2f GB, far above the 126 MB L2" % (
                (w.T * w.H * 2 * 2 + w.T * w.k * w.H * ((1 if w.fp8 else 2) + (1 if w.fp8_combine else 2))) / 1e9),
            "parallelism": f"dp{world}"}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch

    from combine_moe_gate_warp_gb300 import workloads
    if args.workload == "all":
        args = argparse.Namespace(**{**vars(args), "workload": HEADLINE_WORKLOAD})
    w = resolve_workload(args)
    inputs = workloads.make_inputs(w, "cpu")
    hi = dict(logits=inputs["logits"].numpy(),
              x=inputs["x"].view(torch.int16).numpy().view(np.uint16))
    if inputs["shared"] is not None:
        hi["shared"] = inputs["shared"].view(torch.int16).numpy().view(np.uint16)
    # seeded expert outputs for the sampled rows
    hi["eo"] = workloads.make_expert_out(w, min(w.r_max, HOST_EO_ROWS), "cpu").view(torch.int16).numpy().view(np.uint16)
    # size one step so that warmup + steps stay within about three minutes
    budget_s = 180.0 / max(1, args.steps + args.warmup)
    T_max = max_sample_tokens(w)
    T_s = min(T_max, 64)
    dt = oracle_sample_run(w, hi, T_s)
    while dt < 0.5 * budget_s and T_s < T_max:
        T_s = min(T_max, max(T_s * 2, int(T_s * budget_s / max(dt, 1e-6) * 0.7)))
        dt = oracle_sample_run(w, hi, T_s)
    for _ in range(args.warmup):
        oracle_sample_run(w, hi, T_s)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_sample_run(w, hi, T_s)
    value = T_s * args.steps / total
    sample = f"first {T_s} of {w.T} tokens of {w.name} per step, single-threaded C oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64 (CPU)",
            "data": "synthetic (seeded), same recipe as the GPU arm", "config": config_of(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import gc

    import torch

    from combine_moe_gate_warp_gb300 import build
    world, rank, local = dist_env()
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build()
    if args.workload == "all":
        names, headline = list(DEFAULT_WORKLOADS), HEADLINE_WORKLOAD
    else:
        names, headline = [args.workload], args.workload
    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
    except Exception:
        bus = None
    sampler = ClockSampler(bus) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    entries = {}
    for name in names:
        wa = argparse.Namespace(**{**vars(args), "workload": name})
        cpu_s = args.cpu_seconds if name == headline else args.cpu_seconds_other
        entries[name] = measure_workload(wa, world, rank, dev, sampler, cpu_s)
        gc.collect()
        torch.cuda.empty_cache()
    if sampler:
        sampler.stop()
    if rank == 0:
        line = dict(entries[headline])
        if len(names) > 1:
            line["headline_workload"] = (f"{headline}: the largest of the workloads timed here (the metric names "
                                         "no workload); every workload's full entry is under 'workloads'")
            line["workloads"] = {n: {k2: v for k2, v in e.items() if k2 not in LINE_ONLY_KEYS}
                                 for n, e in entries.items()}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# keys of the contract line that a per-workload entry does not repeat
LINE_ONLY_KEYS = ("metric", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline",
                  "data")


def measure_workload(args, world, rank, dev, sampler, cpu_seconds):
    """Every measurement of one workload: the timed one-stream steps (with
    per-call events on every 8th step), the pipelined batches and the CUDA
    graph replays (the headline takes the fastest), the data-movement calls
    back to back for the roofline, the combine's ulp statistics, end to end
    from host buffers, the de-duplicated send path, the backward calls and
    the oracle's CPU baseline.  Returns the workload's JSON entry."""
    import torch

    from combine_moe_gate_warp_gb300 import RoutePipeline, RoutePlan, RouteShape, workloads
    w = rank_workload(resolve_workload(args), rank)

    inputs = workloads.make_inputs(w, dev)
    shape = RouteShape(T=w.T, H=w.H, E=w.E, k=w.k, P=w.P, mode=w.mode, fp8=int(w.fp8), Ks=w.Ks,
                       capacity=w.capacity, fp8_combine=int(w.fp8_combine), reassign=bool(w.reassign))
    plan = RoutePlan(shape, dev)
    eo = None if w.identity_experts else workloads.make_expert_out(w, max(plan.r_max, 1), dev)
    stream = torch.cuda.current_stream(dev)
    eo_arg = plan.packed if eo is None else eo

    for _ in range(max(3, args.warmup)):
        plan.step(inputs["logits"], inputs["x"], eo_arg, inputs["shared"])
    torch.cuda.synchronize(dev)
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"{w.name}: device status {st} after warm-up")
    R = int(plan.layout.offsets[w.E].item())

    K = args.steps
    EV = 8  # per-call CUDA events on every EV-th step (events between kernels cost ~10 us/step)
    sampled = list(range(0, K, EV))
    if plan.fused_route:
        calls = [("route", lambda: plan.route(inputs["logits"]))]
    else:
        calls = [("gate", lambda: plan.gate(inputs["logits"])), ("layout", plan.dispatch_layout)]
    calls += [("dispatch", lambda: plan.dispatch(inputs["x"]))]
    if w.fp8_combine:
        calls += [("quantize", lambda: plan.quantize_expert_out(eo_arg)),
                  ("combine", lambda: plan.combine_fp8(inputs["shared"]))]
    else:
        calls += [("combine", lambda: plan.combine(eo_arg, inputs["shared"]))]
    names = [c[0] for c in calls]
    ev = {i: [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for i in sampled}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(K):
        e = ev.get(i)
        if e is None:
            plan.step(inputs["logits"], inputs["x"], eo_arg, inputs["shared"])
            continue
        e[0].record(stream)
        for j, (n, fn) in enumerate(calls):
            torch.cuda.nvtx.range_push(n)
            fn()
            torch.cuda.nvtx.range_pop()
            e[j + 1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_wall1 = time.time()
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"{w.name}: device status {st} during the timed steps")
    # the combine's accuracy on the last timed step's output
    ulp = combine_ulp_stats(plan, w, eo_arg, inputs["shared"])
    pipe = None
    t_pw0 = t_pw1 = None
    if not args.no_pipeline and RoutePipeline.overlaps(shape):
        runs = []
        configs = PIPE_CONFIGS if args.data_streams == 0 else ((2, args.data_streams),)
        for depth, ds in configs:
            t0 = time.time()
            r = time_pipelined(w, shape, inputs, eo, dev, world, K, max(3, args.warmup), args.route_priority, ds,
                               depth)
            r["depth"], r["data_streams"] = depth, ds
            runs.append((r, t0, time.time()))
            torch.cuda.empty_cache()
        pipe, t_pw0, t_pw1 = min(runs, key=lambda x: x[0]["ms_per_step"])
        if len(runs) > 1:
            pipe["configs_ms"] = {f"plans {r['depth']}, data streams {r['data_streams']}": r["ms_per_step"]
                                  for r, _, _ in runs}
    graph = None
    if not args.no_graph:
        t_gw0 = time.time()
        graph = time_graph(w, shape, inputs, eo, dev, world, K, max(3, args.warmup))
        t_gw1 = time.time()
    per = {n: statistics.fmean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in sampled)
           for j, n in enumerate(names)}
    step_samples = sorted(ev[i][0].elapsed_time(ev[i][len(calls)]) for i in sampled)
    by = kernel_bytes(w, R)
    peak, peak_kind = hbm_peak()
    # the data-movement calls once more, each alone: B2B launches back to back
    # between two events on their stream (no event between launches, so the
    # programmatic launch overlap is kept and the mean is the launch duration)
    B2B = 50
    b2b = {}
    for n, fn in calls:
        if n not in ("dispatch", "quantize", "combine"):
            continue
        for _ in range(3):
            fn()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(B2B):
            fn()
        a1.record(stream)
        torch.cuda.synchronize(dev)
        b2b[n] = a0.elapsed_time(a1) / B2B
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"{w.name}: device status {st} in the back-to-back launches")
    dom = max(("dispatch", "combine"), key=lambda n: b2b[n])
    achieved = by[dom] / (b2b[dom] * 1e-3) / 1e9
    achieved_ev = by[dom] / (per[dom] * 1e-3) / 1e9
    traffic = measured_traffic(dom, w.name, w)
    ms_step_serial = elapsed_ms / K
    unpipelined = {"ms_per_step": ms_step_serial,
                   "tokens_per_s": world * w.T * K / (elapsed_ms * 1e-3),
                   "hbm_frac": by["roofline_step"] / (ms_step_serial * 1e-3) / 1e9 / peak,
                   "note": "the calls of each step on one stream, one batch after another"}
    # the headline is the fastest of the product's ways to run the same steps
    modes = [(ms_step_serial, unpipelined["note"], (t_wall0, t_wall1))]
    if pipe:
        pipe["hbm_frac"] = by["roofline_step"] / (pipe["ms_per_step"] * 1e-3) / 1e9 / peak
        modes.append((pipe["ms_per_step"], pipe["note"], (t_pw0, t_pw1)))
    if graph:
        modes.append((graph["ms_per_step"], graph["note"], (t_gw0, t_gw1)))
        graph["tokens_per_s"] = world * w.T / (graph["ms_per_step"] * 1e-3)
        graph["hbm_frac"] = by["roofline_step"] / (graph["ms_per_step"] * 1e-3) / 1e9 / peak
    ms_step, execution, (t_h0, t_h1) = min(modes, key=lambda m: m[0])
    tokens_per_s = world * w.T / (ms_step * 1e-3)
    step_gbs = by["roofline_step"] / (ms_step * 1e-3) / 1e9

    # end to end through the public API: pinned host inputs copied in, result copied out
    e2e = None
    if not args.no_e2e:
        e2e = time_e2e(w, shape, plan, inputs, eo, dev, world, args.e2e_steps, pipe is not None, R,
                       pipe["data_streams"] if pipe else 1, pipe["depth"] if pipe else 2)

    dd = None
    if args.dedup_steps > 0 and 1 <= w.P <= 16:
        dd = time_dedup(plan, w, inputs, args.dedup_steps, world, dev, stream, peak, R)

    bwd = None
    if args.backward_steps > 0:
        bwd = time_backward(plan, w, inputs, eo_arg, args.backward_steps, world, dev, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, host_inputs(w, inputs, eo), cpu_seconds, args.oracle_threads)

    clocks = sampler.summary(t_h0, t_h1) if sampler else None
    return {
        "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if w.fp8 else "bf16",
        "data": "synthetic (seeded): x ~ N(0,1) bf16, router logits fp32, expert outputs N(0,1) bf16",
        "config": config_of(w, world),
        "hbm_gbs": step_gbs, "hbm_frac": step_gbs / peak, "R": R,
        "hbm_gbs_all_bytes": by["all_step"] / (ms_step * 1e-3) / 1e9,
        "hbm_frac_all_bytes": by["all_step"] / (ms_step * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes": by[dom], "launch_ms": b2b[dom],
                     "timing": f"mean of {B2B} back-to-back launches of the call between CUDA events "
                               "on its stream, after the timed steps",
                     "achieved_evented": achieved_ev, "frac_evented": achieved_ev / peak,
                     "launch_ms_evented": per[dom],
                     "timing_evented": "mean over the sampled timed steps with CUDA events around each call "
                                       "(includes the launch gap the events add)"},
        "kernels_ms_back_to_back": b2b,
        "kernels_ms": per,
        "kernels_sampled_steps": len(sampled),
        "kernels_gbs": {n: by[n] / (per[n] * 1e-3) / 1e9 for n in names},
        "step_ms_evented": {"median": statistics.median(step_samples), "min": step_samples[0],
                            "note": "sampled steps with events between the calls"},
        "execution": execution,
        "unpipelined": unpipelined,
        "pipelined": pipe,
        "graph": graph,
        "gpu_launches": plan.launches_per_step() * K,
        "clocks": clocks,
        "combine_ulp": ulp,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "backward": bwd,
        "dedup": dd,
    }


def combine_ulp_stats(plan, w, eo, shared):
    """How many combine outputs of the last step lie beyond one bf16 ulp of
    the fp64 sum of their terms (the same gates, rows and shared outputs the
    kernel read), and the largest share of the fp32 summation allowance
    n * 2^-24 * sum|terms| that such an output uses (above 1 would be outside
    the bound the tests enforce).  Computed on the GPU in fp64 with torch,
    in token chunks."""
    import torch
    T, k, H, Ks = w.T, w.k, w.H, w.Ks
    if T == 0:
        return {"outputs": 0, "beyond_1ulp": 0, "outside_bound": 0, "max_allowance_used": 0.0}
    dst = plan.layout.dst_row[:T * k].view(T, k).long()
    g = plan.gates[:T].double()
    n_terms = k + Ks + (1 if w.fp8_combine else 0)
    if w.fp8_combine:
        vals = plan.eo_codes.view(torch.float8_e4m3fn)
        sc = plan.eo_scales.double()
    chunk = max(1, (1 << 24) // max(1, H))
    beyond = outside = 0
    used = 0.0
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        acc = torch.zeros((t1 - t0, H), dtype=torch.float64, device=g.device)
        mag = torch.zeros_like(acc)
        for j in range(k):
            r = dst[t0:t1, j]
            keep = (r >= 0).double().unsqueeze(1)
            rr = r.clamp(min=0)
            if w.fp8_combine:
                # the dequantised row is rounded to fp32 once, as the kernel does
                rows = (vals.index_select(0, rr).double() * sc[rr, 0:1] + sc[rr, 1:2]).float().double()
            else:
                rows = eo.index_select(0, rr).double()
            term = rows * g[t0:t1, j:j + 1] * keep
            acc += term
            mag += term.abs()
        for s_ in range(Ks):
            term = shared[s_, t0:t1].double()
            acc += term
            mag += term.abs()
        err = (plan.y[t0:t1].double() - acc).abs()
        _, ex = torch.frexp(acc)
        e = torch.where(acc == 0, torch.full_like(ex, -200), ex - 1).clamp(min=-126)
        ulp = torch.pow(2.0, (e - 7).double())
        allow = n_terms * 2.0 ** -24 * mag
        over = err > ulp
        beyond += int(over.sum().item())
        outside += int((err > ulp + allow).sum().item())
        if bool(over.any()):
            used = max(used, float(((err - ulp)[over] / allow[over].clamp(min=1e-300)).max().item()))
    return {"outputs": T * H, "beyond_1ulp": beyond, "beyond_1ulp_frac": beyond / (T * H),
            "outside_bound": outside, "max_allowance_used": used,
            "how": "each y against the fp64 sum of its terms (the kernel's gates, rows and shared outputs), "
                   "on the GPU; allowance n * 2^-24 * sum|terms| with n = the number of terms"}


def time_e2e(w, shape, plan, inputs, eo, dev, world, steps, pipelined, R, data_streams=2, depth=2):
    """The same metric end to end: every step copies its inputs (router
    logits, x, the R expert-output rows the batch produces, shared-expert
    outputs) from pinned host memory to the device and reads y, the aux loss
    and the entropy back.  With the pipelined executor the copies of batch
    i+1 overlap the work of batch i (a copy stream feeds each plan's own
    input buffers); otherwise the copies and the calls run in order on one
    stream.  (Every step routes the same batch, so R is the warm-up's.)"""
    import torch

    from combine_moe_gate_warp_gb300 import RoutePipeline
    pin = dict(logits=inputs["logits"].cpu().pin_memory(), x=inputs["x"].cpu().pin_memory())
    eo_h = None if eo is None else eo[:max(R, 1)].cpu().pin_memory()
    sh_h = None if inputs["shared"] is None else inputs["shared"].cpu().pin_memory()
    y_h = torch.empty((w.T, w.H), dtype=torch.bfloat16, pin_memory=True)
    stats_h = torch.empty(2, dtype=torch.float64, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (pin["logits"], pin["x"], eo_h, sh_h) if t is not None)
    d2h = y_h.numel() * y_h.element_size() + 16

    def dev_buffers():
        return dict(logits=torch.empty_like(inputs["logits"]), x=torch.empty_like(inputs["x"]),
                    eo=None if eo is None else torch.empty_like(eo),
                    shared=None if inputs["shared"] is None else torch.empty_like(inputs["shared"]))

    def copy_in(d):
        d["logits"].copy_(pin["logits"], non_blocking=True)
        d["x"].copy_(pin["x"], non_blocking=True)
        if d["eo"] is not None:
            d["eo"][:eo_h.shape[0]].copy_(eo_h, non_blocking=True)
        if d["shared"] is not None:
            d["shared"].copy_(sh_h, non_blocking=True)

    K2 = max(1, steps)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pipelined:
        pipe = RoutePipeline(shape, dev, depth=depth, data_streams=data_streams)
        bufs = [dev_buffers() for _ in pipe.plans]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in pipe.plans]

        def one():
            i = pipe.step_index
            d = i % len(pipe.plans)
            copy_stream.wait_event(pipe.release_event(i))
            with torch.cuda.stream(copy_stream):
                copy_in(bufs[d])
            copied[d].record(copy_stream)
            pipe.route_stream.wait_event(copied[d])
            pipe.stream_for(i).wait_event(copied[d])
            p = pipe.plan_for(i)
            bd = bufs[d]
            pipe.step(bd["logits"], bd["x"], p.packed if bd["eo"] is None else bd["eo"], bd["shared"],
                      out=y_h, stats_out=stats_h)

        for _ in range(3):
            one()
        pipe.synchronize()
        barrier(world)
        torch.cuda.synchronize(dev)
        a.record(copy_stream)
        pipe.wait_event(a)
        for _ in range(K2):
            one()
        pipe.record(b)
        torch.cuda.synchronize(dev)
        st = pipe.status()
        path = ("pinned host -> device copies on a copy stream into each plan's input buffers, the C-ABI "
                "calls through RoutePipeline, y/aux/entropy back on the data stream; batch i+1's copies "
                "and routing overlap batch i's data movement")
    else:
        stream = torch.cuda.current_stream(dev)
        d = dev_buffers()

        def one():
            copy_in(d)
            plan.step(d["logits"], d["x"], plan.packed if d["eo"] is None else d["eo"], d["shared"])
            y_h.copy_(plan.y[:w.T], non_blocking=True)
            stats_h[0:1].copy_(plan.aux_loss, non_blocking=True)
            stats_h[1:2].copy_(plan.entropy, non_blocking=True)

        for _ in range(3):
            one()
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(K2):
            one()
        b.record(stream)
        torch.cuda.synchronize(dev)
        st = plan.status()
        path = "pinned host -> device copies, the C-ABI calls, y/aux/entropy back, one stream"
    if st != 0:
        raise RuntimeError(f"device status {st} in the end-to-end steps")
    e_ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": world * w.T * K2 / (e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / K2, "steps": K2, "path": path}


def pipe_streams(pipe) -> int:
    return len(getattr(pipe, "data_streams", [pipe.data_stream]))


# RoutePipeline configurations the bench times (plans, data streams); the
# fastest is the pipelined figure
PIPE_CONFIGS = ((2, 1), (2, 2), (3, 3))


def time_pipelined(w, shape, inputs, eo, dev, world, K, W, route_priority="high", data_streams=2, depth=2):
    """K back-to-back batches through RoutePipeline: two plans and two input
    batches (the workload's seed and the next one) alternate, so every step
    routes a batch while the previous batch's dispatch and combine run."""
    import torch

    from combine_moe_gate_warp_gb300 import RoutePipeline, workloads
    w2 = workloads.Workload(**{**w.__dict__, "seed": w.seed + 1})
    inputs2 = workloads.make_inputs(w2, dev)
    pipe = RoutePipeline(shape, dev, depth=depth, route_priority=route_priority, data_streams=data_streams)
    eo2 = None if eo is None else workloads.make_expert_out(w2, max(pipe.plans[0].r_max, 1), dev)
    batches = [(inputs, eo), (inputs2, eo2)]

    def one(i):
        inp, e = batches[i % 2]
        p = pipe.plan_for(pipe.step_index)
        pipe.step(inp["logits"], inp["x"], p.packed if e is None else e, inp["shared"])

    torch.cuda.synchronize(dev)
    for i in range(W):
        one(i)
    torch.cuda.synchronize(dev)
    st = pipe.status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the pipelined warm-up")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    start.record(pipe.data_stream)
    pipe.wait_event(start)
    for i in range(K):
        one(W + i)
    pipe.record(stop)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(stop), world, dev) / K
    st = pipe.status()
    if st != 0:
        raise RuntimeError(f"device status {st} during the pipelined steps")
    return {"ms_per_step": ms,
            "note": "back-to-back batches (two alternating input batches, %d plans): the routing of batch "
                    "i on a high-priority stream overlaps the data calls of the batches before it; the data "
                    "calls of consecutive batches on %d alternating streams" % (len(pipe.plans), pipe_streams(pipe))}


def time_graph(w, shape, inputs, eo, dev, world, K, W):
    """K replays of the one-stream step captured as a CUDA graph
    (RouteGraph): inputs loaded into the graph's buffers once, then
    replayed back to back between two events on the graph's stream."""
    import torch

    from combine_moe_gate_warp_gb300 import RouteGraph
    g = RouteGraph(shape, dev)
    g.step(inputs["logits"], inputs["x"], eo, inputs["shared"])
    for _ in range(W):
        g.replay()
    torch.cuda.synchronize(dev)
    st = g.status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the graph warm-up")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    start.record(g.stream)
    for _ in range(K):
        g.replay()
    stop.record(g.stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(stop), world, dev) / K
    st = g.status()
    if st != 0:
        raise RuntimeError(f"device status {st} during the graph replays")
    return {"ms_per_step": ms, "launches_per_step": g.launches_per_step(),
            "note": "the calls of each step on one stream, captured once as a CUDA graph and replayed"
                    + (" (identity experts: the graph's expert-output buffer stands in for the packed rows)"
                       if eo is None else "")}


def time_dedup(plan, w, inputs, steps, world, dev, stream, peak, R):
    """The per-partition de-duplicated send path on the forward's layout:
    moe_dedup_layout (send rows) and moe_dispatch_dedup (x copied once per
    partition a token reaches).  Reports the send rows against the packed
    rows (what an expert-parallel exchange would move) and the times."""
    import torch

    from combine_moe_gate_warp_gb300 import abi
    D = abi.Dedup(w.T, w.k, w.P, dev)
    fp8 = 1 if int(w.fp8) == 1 else 0
    send = torch.empty((D.s_max, w.H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    sc = torch.empty((D.s_max, 2), dtype=torch.float32, device=dev) if fp8 else None

    def one(e=None):
        if e:
            e[0].record(stream)
        abi.moe_dedup_layout(plan.layout, plan.gates, D, stream)
        if e:
            e[1].record(stream)
        abi.moe_dispatch_dedup(inputs["x"], w.T, w.H, D, fp8, send, sc, stream)
        if e:
            e[2].record(stream)

    for _ in range(3):
        one()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(world)
    for e in ev:
        one(e)
    torch.cuda.synchronize(dev)
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"device status {st} in the de-duplicated path")
    S = int(D.send_offsets[w.P].item())
    t_lay = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev)
    t_disp = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev)
    bt = 1 if fp8 else 2
    disp_bytes = w.T * w.H * 2 + S * w.H * bt + (S * 8 if fp8 else 0)
    # send rows when the experts are grouped by rank of an expert-parallel
    # exchange of W ranks (one group per rank: a token goes to a rank once)
    by_ranks = {}
    for g in (2, 4, 8, 16):
        if g > w.E or w.E % g:
            continue
        Dg = abi.Dedup(w.T, w.k, g, dev)
        abi.moe_dedup_layout(plan.layout, plan.gates, Dg, stream, groups=g)
        Sg = int(Dg.send_offsets[g].item())
        by_ranks[str(g)] = {"send_rows": Sg, "send_over_packed": Sg / max(R, 1),
                            "bytes_saved_per_step": (R - Sg) * w.H * bt * 2}
        del Dg
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"device status {st} in the de-duplicated layouts per rank group")
    return {"send_rows": S, "packed_rows": R, "send_over_packed": S / max(R, 1),
            "layout_ms": t_lay, "dispatch_ms": t_disp,
            "dispatch_gbs": disp_bytes / (t_disp * 1e-3) / 1e9,
            "dispatch_frac": disp_bytes / (t_disp * 1e-3) / 1e9 / peak, "steps": steps,
            "by_ranks": by_ranks,
            "by_ranks_note": "send rows with the experts grouped per rank of a W-rank exchange (W = key); "
                             "bytes saved per step count both directions (rows out, partial rows back)"}


def time_backward(plan, w, inputs, eo_arg, steps, world, dev, stream, peak):
    """The backward calls on the forward's layout, timed after the forward
    (not part of the headline step): combine backward (d_expert_out,
    d_gates), gate backward (d_logits) and dispatch backward (dx).  Returns
    per-kernel times, algorithmic-byte throughput and roofline fractions."""
    import torch

    from combine_moe_gate_warp_gb300 import workloads
    R = int(plan.layout.offsets[w.E].item())
    dy = workloads.make_dy(w, dev)
    dp = workloads.make_d_packed(w, max(plan.r_max, 1), dev)
    for _ in range(3):
        plan.backward(inputs["logits"], dy, eo_arg, dp)
    torch.cuda.synchronize(dev)
    names = ["combine_backward", "gate_backward", "dispatch_backward"]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    torch.cuda.nvtx.range_push("backward")  # a profiler can select these launches by range
    for e in ev:
        e[0].record(stream)
        plan.combine_backward(dy, eo_arg)
        e[1].record(stream)
        plan.gate_backward(inputs["logits"])
        e[2].record(stream)
        plan.dispatch_backward(dp)
        e[3].record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    per = {n: statistics.fmean(e[j].elapsed_time(e[j + 1]) for e in ev) for j, n in enumerate(names)}
    # whole backward without events between the kernels
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        plan.backward(inputs["logits"], dy, eo_arg, dp)
    b.record(stream)
    torch.cuda.synchronize(dev)
    total_ms = max_over_ranks(a.elapsed_time(b) / steps, world, dev)
    st = plan.status()
    if st != 0:
        raise RuntimeError(f"device status {st} during the backward passes")
    by = workloads.nbytes_backward(w, R)
    gbs = {n: by[n] / (per[n] * 1e-3) / 1e9 for n in names}
    return {"steps": steps, "ms_per_pass": total_ms,
            "traffic": {n: measured_traffic(n, w.name, w) for n in names},
            "tokens_per_s": world * w.T / (total_ms * 1e-3),
            "kernels_ms": per, "kernels_gbs": gbs,
            "kernels_frac": {n: gbs[n] / peak for n in names},
            "algorithmic_bytes": by, "gpu_launches": 3 * steps * 2}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
