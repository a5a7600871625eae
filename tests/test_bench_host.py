"""Host logic of bench.py (no GPU): the algorithmic byte counts behind the
roofline fractions, and the rule that measured DRAM traffic is reported only
for the kernel source it was taken on."""
import importlib.util
import json
import os
import sys

import pytest

from combine_moe_gate_warp_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_v2_top2_step_bytes(bench):
    """16384 tokens x 5120 bf16, top-2, no capacity (R = T k = 32768): x read
    and y written once (167.8 MB each), packed rows written and expert rows
    read once (335.5 MB each): 61440 bytes per token, 1.0066 GB per step."""
    w = workloads.WORKLOADS["v2_top2"]
    R = w.T * w.k
    by = bench.kernel_bytes(w, R)
    x = 16384 * 5120 * 2
    assert by["dispatch"] == x + R * 5120 * 2
    assert by["combine"] == R * 5120 * 2 + x + w.T * w.k * 8
    assert by["roofline_step"] == 61440 * 16384 == 1006632960
    assert by["roofline_step"] == workloads.nbytes_roofline(w, R)


def test_fp8_and_shared_expert_bytes(bench):
    """Per-token e4m3 transport: one byte per packed element plus the (scale,
    zero) pair per row; grouped modes read x twice; shared experts add their
    rows to the combine's reads but not to the metric's bytes."""
    w = workloads.WORKLOADS["fp8_skewed"]
    R = w.T * w.k
    by = bench.kernel_bytes(w, R)
    assert by["dispatch"] == w.T * w.H * 2 + R * w.H + R * 8
    ge = workloads.WORKLOADS["fp8_expert"]
    assert bench.kernel_bytes(ge, R)["dispatch"] == 2 * w.T * w.H * 2 + R * w.H + R * 8
    fs = workloads.WORKLOADS["fine_shared"]
    Rf = fs.T * fs.k
    byf = bench.kernel_bytes(fs, Rf)
    assert byf["combine"] - (Rf * fs.H * 2 + fs.T * fs.H * 2 + fs.T * fs.k * 8) == 2 * fs.T * fs.H * 2
    assert byf["roofline_step"] == workloads.nbytes_roofline(fs, Rf)


def test_traffic_only_for_the_source_it_was_taken_on(bench, monkeypatch):
    """measured_traffic gives the committed DRAM bytes while the kernel's
    sources hash to the digest stored with them, and None otherwise (or for
    a workload the table does not hold)."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        table = json.load(f)
    wl, kern = "v2_top2", "combine"
    ent = table[wl][kern]
    w = workloads.WORKLOADS[wl]
    monkeypatch.setattr(bench, "source_digest", lambda name, w=None: ent["source_digest"])
    assert bench.measured_traffic(kern, wl, w) == ent["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "source_digest", lambda name, w=None: "0" * 16)
    assert bench.measured_traffic(kern, wl, w) is None
    assert bench.measured_traffic(kern, "no_such_workload", w) is None


def test_source_digest_follows_the_kernel_files(bench):
    """Each call's digest covers the files its kernel is built from: the
    bf16 and FP8 dispatches hash different sources."""
    v2 = workloads.WORKLOADS["v2_top2"]
    f8 = workloads.WORKLOADS["fp8_skewed"]
    assert "dispatch.cu" in bench.kernel_sources("dispatch", v2)
    assert "quant.cu" in bench.kernel_sources("dispatch", f8)
    assert bench.source_digest("dispatch", v2) != bench.source_digest("dispatch", f8)
    assert bench.source_digest("combine", v2) == bench.source_digest("combine", f8)
