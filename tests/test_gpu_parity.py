"""GPU parity: the CUDA path, called through the C ABI, against the CPU
oracle on the same seeded inputs.

Bit-exact: top-k ids, counts, offsets, permutation, capacity drops, packed
bf16 rows, FP8 codes and scales, and the combine in its pinned fp32 order.
Gate weights within 1e-6 absolute (fp32 vs the fp64 oracle); aux loss and
entropy within 1e-9 and 1e-6 (fp64 from the same integer counts; the entropy uses fp32 mantissa logarithms); the combine also
within one bf16 ulp of the fp64 reference plus the fp32 summation bound.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import workloads
from gpu_util import (bits, check_combine, check_combine_full, check_dispatch, check_dispatch_full, check_gate,
                      check_layout, route_checked, run_gpu)

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()
    torch.cuda.init()


def _full_check(w, seed=7, fused=None):
    """Gate, layout, every packed row and every output token of workload w
    against the oracle; returns the plan, the oracle layout and the
    beyond-one-ulp statistics of the combine.  fused: routing by moe_route
    (default where it applies) or by moe_gate + the layout call (False)."""
    inp = workloads.make_inputs(w, "cuda")
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp, fused=fused)
    assert status == 0, f"device status {status}"
    idx, counts = check_gate(w, plan, gates_pre, og)
    assert counts.sum() == w.T * w.k
    L = check_layout(w, plan, og)
    assert L["R"] == R
    x_bits = bits(inp["x"])
    check_dispatch_full(w, plan, L, x_bits)
    st = check_combine_full(w, plan, L, eo, inp["shared"], x_bits)
    assert st.outputs == w.T * w.H
    return plan, L, st


# --- small cases: every output compared element by element ----------------
# Token counts span several gate/layout tiles with a ragged tail.
SMALL = [
    W["tiny"],
    W["v2_top2"].scaled(1000),
    W["fine_shared"].scaled(333),
    W["fp8_skewed"].scaled(1500),
    W["prefill_cap"].scaled(700),
]


ROUTING = [pytest.param(True, id="moe_route"), pytest.param(False, id="gate+layout")]


@pytest.mark.parametrize("fused", ROUTING)
@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_workloads_exact(w, fused):
    plan, L, st = _full_check(w, fused=fused)
    if w.identity_experts:
        assert np.array_equal(bits(plan.y), bits(workloads.make_x(w, "cuda")))


# --- the full-size workloads: every output compared, in chunks ------------
@pytest.mark.parametrize("name", ["tiny", "v2_top2", "fine_shared", "fp8_skewed", "prefill_cap"])
def test_full_size_workloads(name):
    w = W[name]
    plan, L, st = _full_check(w)
    if name == "prefill_cap":
        assert L["dropped"] > 0 and np.all(L["counts"] <= w.capacity)


@pytest.mark.parametrize("name", ["v2_top2", "fine_shared", "fp8_skewed", "prefill_cap"])
def test_full_size_gate_and_layout_calls(name):
    """The separate moe_gate and moe_dispatch_layout calls at full size (the
    dispatch and combine do not depend on which routing call ran)."""
    from combine_moe_gate_warp_gb300 import RoutePlan
    from gpu_util import gate_with_oracle, poison, shape_of
    w = W[name]
    inp = workloads.make_inputs(w, "cuda")
    plan = RoutePlan(shape_of(w), "cuda")
    plan.fused_route = False
    poison(plan)
    gates_pre, og = gate_with_oracle(w, plan, inp["logits"])
    plan.dispatch_layout()
    assert plan.status() == 0
    check_gate(w, plan, gates_pre, og)
    check_layout(w, plan, og)


# --- edge cases --------------------------------------------------------------
def _custom(T, H, E, k, P, mode=0, fp8=False, Ks=0, cap_factor=0.0, seed=99, **kw):
    return workloads.Workload(f"edge_T{T}_E{E}_k{k}", T=T, H=H, E=E, k=k, P=P, mode=mode, fp8=fp8, Ks=Ks,
                              capacity_factor=cap_factor, seed=seed, **kw)


EDGE = [
    _custom(1, 8, 8, 2, 4),                    # one token, smallest H
    _custom(3, 16, 8, 8, 8),                   # k == E
    _custom(257, 64, 256, 16, 256),            # largest E and k, one expert per partition
    _custom(2049, 24, 5, 3, 1, mode=1),        # odd E, P = 1, many tiles
    _custom(129, 16, 8, 1, 2, fp8=True),       # k = 1, smallest FP8 row
    _custom(300, 8200, 16, 2, 4),              # H > 8192: looped copy
    _custom(64, 16384, 8, 2, 2, fp8=True),     # largest FP8 row
    _custom(500, 40, 12, 4, 3, Ks=3, mode=1),  # ragged H / 8, three shared experts
]


@pytest.mark.parametrize("fused", ROUTING)
@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edge_shapes(w, fused):
    _full_check(w, fused=fused)


@pytest.mark.parametrize("fused", ROUTING)
def test_empty_batch(fused):
    w = _custom(0, 64, 8, 2, 4)
    inp = workloads.make_inputs(w, "cuda")
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp, fused=fused)
    assert status == 0 and R == 0
    assert plan.expert_counts.cpu().tolist() == [0] * 8
    assert plan.aux_loss.item() == 0.0 and plan.entropy.item() == 0.0
    assert plan.layout.offsets.cpu().tolist() == [0] * 9
    assert plan.layout.part_tokens.cpu().tolist() == [0] * 4


def _run_with_logits(w, logits, fused=None):
    inp = dict(logits=logits.contiguous(), x=workloads.make_x(w, "cuda"), shared=None)
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp, fused=fused)
    assert status == 0
    check_gate(w, plan, gates_pre, og)
    L = check_layout(w, plan, og)
    check_dispatch(w, plan, L, bits(inp["x"]), np.arange(R, dtype=np.int64))
    check_combine(w, plan, L, eo, None, np.arange(w.T, dtype=np.int64), bits(inp["x"]))
    return plan, L


@pytest.mark.parametrize("fused", ROUTING)
def test_ties_and_signed_zeros(fused):
    w = _custom(1100, 32, 16, 4, 4)
    g = torch.Generator(device="cuda").manual_seed(5)
    logits = torch.randint(-2, 3, (w.T, w.E), generator=g, device="cuda").float()
    logits[torch.rand((w.T, w.E), generator=g, device="cuda") < 0.2] = -0.0
    _run_with_logits(w, logits, fused)


# Gate shapes through the one-thread-per-token gate: k not a power of two,
# long rows (E = 96, 256) staged with 16-byte loads, E % 4 != 0 (4-byte
# staging loads), a ragged last tile, the SOFTMAX_TOPK mode, and more tokens
# than the GPU holds resident threads.
GATE_SHAPES = [
    _custom(3001, 16, 96, 6, 8),                # k = 6 of 96
    _custom(1201, 16, 256, 5, 8, mode=1),       # E = 256, softmax over all E
    _custom(999, 16, 20, 3, 4),                 # E = 20, ragged last tile
    _custom(777, 16, 6, 2, 2, mode=1),          # E = 6: 4-byte staging loads
    _custom(200003, 16, 64, 2, 8),              # more tokens than resident threads
]


@pytest.mark.parametrize("fused", ROUTING)
@pytest.mark.parametrize("w", GATE_SHAPES, ids=[w.name for w in GATE_SHAPES])
@pytest.mark.parametrize("ties", [False, True])
def test_gate_shapes(w, ties, fused):
    if ties:
        g = torch.Generator(device="cuda").manual_seed(w.E)
        logits = torch.randint(-2, 3, (w.T, w.E), generator=g, device="cuda").float()
        logits[torch.rand((w.T, w.E), generator=g, device="cuda") < 0.2] = -0.0
    else:
        logits = workloads.make_inputs(w, "cuda")["logits"]
    _run_with_logits(w, logits, fused)


@pytest.mark.parametrize("fused", ROUTING)
def test_ties_large_k(fused):
    """Integer logits in {-1, 0, 1} with signed zeros and k up to 16: most of
    a token's list is made of equal values, so the insertion order decides
    every position (ties to the lower expert id, -0 == +0)."""
    for E, k in ((64, 8), (256, 16), (128, 4)):
        w = _custom(513, 16, E, k, 8)
        g = torch.Generator(device="cuda").manual_seed(k)
        logits = torch.randint(-1, 2, (w.T, w.E), generator=g, device="cuda").float()
        logits[torch.rand((w.T, w.E), generator=g, device="cuda") < 0.3] = -0.0
        _run_with_logits(w, logits, fused)


class _with_capacity:
    """A workload view with an explicit capacity (the capacity property of
    Workload is derived from its factor)."""

    def __init__(self, w, cap):
        self._w, self.capacity = w, cap

    def __getattr__(self, name):
        return getattr(self._w, name)


def test_all_tokens_one_expert_capacity_hit_exactly_and_exceeded():
    """Every token picks experts 5 then 2; capacity at, one below, and far
    below the per-expert load."""
    from combine_moe_gate_warp_gb300 import RoutePlan
    from gpu_util import shape_of
    w = workloads.Workload("hot", T=1000, H=32, E=8, k=2, P=4, seed=3)
    logits = torch.zeros((w.T, w.E), device="cuda")
    logits[:, 5] = 4.0
    logits[:, 2] = 3.0
    x = workloads.make_x(w, "cuda")
    for cap in (1000, 999, 1):
        shp = shape_of(w)
        shp.capacity = cap
        plan = RoutePlan(shp, "cuda")
        idx = oracle.gate(logits.cpu().numpy(), 2, 0)[0]
        assert np.all(idx == [5, 2])
        # the capacity lives in the plan's shape; the oracle gets the same value
        wc = workloads.Workload("hot", T=1000, H=32, E=8, k=2, P=4, seed=3)
        L = route_checked(_with_capacity(wc, cap), plan, logits)
        plan.dispatch(x)
        assert plan.status() == 0
        assert int(plan.layout.dropped.item()) == 2 * 1000 - 2 * min(cap, 1000)
        check_dispatch(wc, plan, L, bits(x), np.arange(L["R"], dtype=np.int64))


def test_fp8_constant_and_signed_zero_rows():
    w = _custom(6, 32, 8, 2, 4, fp8=True)
    inp = workloads.make_inputs(w, "cuda")
    x = inp["x"]
    x[0] = 0.75                       # constant row
    x[1] = 0.0
    x[1, ::2] = -0.0                  # +-0 mix: max +0, min -0, flat
    x[2] = -0.0                       # all -0: zero word is -0
    x[3, :] = 1.0
    x[3, 7] = -448.0                  # min hits -448 exactly
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp)
    assert status == 0
    check_gate(w, plan, gates_pre, og)
    L = check_layout(w, plan, og)
    check_dispatch(w, plan, L, bits(x), np.arange(R, dtype=np.int64))


def test_fp8_bf16_pattern_sweep():
    """Every finite bf16 value x, placed in rows headed by (M, -M) with
    M = 448 * 2^m, so that (unless x itself exceeds M) scale = 2^m and
    v = x / 2^m is exact; m runs so that v's binary exponent covers
    [-12, 8]: every rounding regime of e4m3 (subnormal ties, normal ties,
    carries into the next binade)."""
    pats = np.arange(65536, dtype=np.uint32)
    f = (pats << 16).view(np.float32)
    pats = pats[np.isfinite(f)]
    f = f[np.isfinite(f)]
    ex = np.where(f == 0, -140, np.floor(np.log2(np.abs(np.where(f == 0, 1, f).astype(np.float64)))))
    vals, heads = [], []
    for s in range(-12, 9):
        m = ex - s
        ok = (m >= -139) & (m <= 118)
        for mm in np.unique(m[ok]):
            sel = pats[ok & (m == mm)]
            M = np.float32(448.0 * 2.0 ** mm)
            Mb = np.uint32(M.view(np.uint32)) >> 16
            assert (np.uint32(Mb) << 16).view(np.float32) == M
            for c in range(0, sel.size, 62):
                vals.append(sel[c:c + 62])
                heads.append(Mb)
    T = len(vals)
    H = 64
    rows = np.zeros((T, H), np.uint16)
    for i, (v, Mb) in enumerate(zip(vals, heads)):
        rows[i, 0] = Mb
        rows[i, 1] = Mb | 0x8000
        rows[i, 2:2 + v.size] = v
        rows[i, 2 + v.size:] = 0
    w = _custom(T, H, 8, 1, 1, fp8=True)
    x = torch.from_numpy(rows.view(np.int16)).cuda().view(torch.bfloat16)
    inp = dict(logits=workloads.make_logits(w, "cuda"), x=x, shared=None)
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp)
    assert status == 0 and R == T
    check_gate(w, plan, gates_pre, og)
    L = check_layout(w, plan, og)
    check_dispatch(w, plan, L, rows, np.arange(R, dtype=np.int64))


@pytest.mark.parametrize("fp8", [1, 3])
def test_fp8_odd_scale_sweep(fp8):
    """Scales 3/128, 5/128, ..., 15/128 (not powers of two: the quotient is
    formed through a reciprocal and checked by the rounding test): rows
    headed by (M, -M) with M = 448 * scale carry every bf16 value in
    [-M, M], so every quotient that lands on an e4m3 rounding midpoint
    exactly, or next to one, is exercised.  Bit-exact against the oracle's
    true division, per-token and global groups."""
    H = 64
    pats = np.arange(65536, dtype=np.uint32)
    f = (pats << 16).view(np.float32)
    rows = []
    for num in (3, 5, 7, 9, 11, 13, 15):
        M = np.float32(448.0 * num / 128.0)
        Mb = np.uint32(M.view(np.uint32)) >> 16
        assert (np.uint32(Mb) << 16).view(np.float32) == M
        vals = pats[np.isfinite(f) & (np.abs(f) <= M)]
        for c in range(0, vals.size, H - 2):
            r = np.zeros(H, np.uint16)
            r[0], r[1] = Mb, Mb | 0x8000
            chunk = vals[c:c + H - 2]
            r[2:2 + chunk.size] = chunk
            rows.append(r)
    rows = np.stack(rows)
    w = _custom(rows.shape[0], H, 8, 1, 1, fp8=fp8)
    x = torch.from_numpy(rows.view(np.int16)).cuda().view(torch.bfloat16)
    inp = dict(logits=workloads.make_logits(w, "cuda"), x=x, shared=None)
    plan, gates_pre, og, R, eo, status = run_gpu(w, inp)
    assert status == 0 and R == w.T
    check_gate(w, plan, gates_pre, og)
    L = check_layout(w, plan, og)
    check_dispatch(w, plan, L, rows, np.arange(R, dtype=np.int64))


def test_repeated_calls_reuse_workspace():
    """The workspace returns to a clean state after every call: three passes
    over different inputs on one plan match fresh oracle runs."""
    from gpu_util import shape_of
    from combine_moe_gate_warp_gb300 import RoutePlan
    w = W["prefill_cap"].scaled(3000)
    plan = RoutePlan(shape_of(w), "cuda")
    for rep in range(3):
        wr = workloads.Workload(**{**w.__dict__, "seed": 500 + rep})
        inp = workloads.make_inputs(wr, "cuda")
        route_checked(wr, plan, inp["logits"])
        plan.dispatch(inp["x"])
        assert plan.status() == 0


def test_mixed_routing_calls_share_a_workspace():
    """moe_route and moe_gate + moe_dispatch_layout alternate on one plan's
    workspace (their cross-block words live in separate regions): every
    call matches the oracle."""
    from combine_moe_gate_warp_gb300 import RoutePlan
    from gpu_util import gate_with_oracle, shape_of
    w = W["prefill_cap"].scaled(6000)
    plan = RoutePlan(shape_of(w), "cuda")
    for rep in range(6):
        wr = workloads.Workload(**{**w.__dict__, "seed": 700 + rep})
        inp = workloads.make_inputs(wr, "cuda")
        plan.fused_route = rep % 2 == 0
        route_checked(wr, plan, inp["logits"])
        plan.dispatch(inp["x"])
        assert plan.status() == 0


@pytest.mark.parametrize("H", [1024, 1032])
@pytest.mark.parametrize("x_off,p_off", [(0, 0), (16, 0), (0, 16), (16, 16)])
def test_dispatch_vector_widths(H, x_off, p_off):
    """The bf16 dispatch moves 32-byte vectors where x, packed and the row
    length (2H bytes) are 32-byte aligned, and 16-byte vectors otherwise:
    both against the oracle, with base pointers 16 bytes past a 32-byte
    boundary and a row of 2064 bytes."""
    from combine_moe_gate_warp_gb300 import RoutePlan, abi
    from gpu_util import shape_of
    w = workloads.Workload("vec", T=777, H=H, E=8, k=3, P=4, seed=11)
    plan = RoutePlan(shape_of(w), "cuda")
    L = route_checked(w, plan, workloads.make_logits(w, "cuda"))
    x0 = workloads.make_x(w, "cuda")
    xb = torch.empty(w.T * H + 16, dtype=torch.bfloat16, device="cuda")
    x = xb[x_off // 2: x_off // 2 + w.T * H].view(w.T, H)
    x.copy_(x0)
    pb = torch.full((plan.r_max * H + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    packed = pb[p_off // 2: p_off // 2 + plan.r_max * H].view(plan.r_max, H)
    assert x.data_ptr() % 32 == x_off and packed.data_ptr() % 32 == p_off
    abi.moe_dispatch(x, w.T, H, plan.layout, 0, packed)
    torch.cuda.synchronize()
    assert plan.status() == 0
    R = int(L["R"])
    src_tok = L["src_pos"].astype(np.int64) // w.k
    assert np.array_equal(bits(packed[:R]), bits(x0)[src_tok])


def test_route_large_batch_resized_tiles():
    """A batch whose 64-token tiles outnumber the blocks the GPU holds at
    once: moe_route doubles the tile until the grid fits, then resizes it to
    ceil(T / resident slots) tokens so every SM holds as many tiles (here
    several gate rounds per tile, the last one partial, and a ragged last
    tile); top-8 of 64 with capacity drops, against the oracle in full."""
    w = workloads.Workload("route_resized", T=120001, H=64, E=64, k=8, P=8, logit_std=1.5, zipf_bias=True,
                           capacity_factor=1.25, seed=52)
    _full_check(w, fused=True)


def test_route_large_batch_many_experts():
    """256 experts (staging rounds of 64 tokens) in a batch whose tiles are
    grown and resized: several gate rounds per tile, the softmax over all
    experts, against the oracle in full."""
    w = workloads.Workload("route_e256", T=100003, H=16, E=256, k=8, P=8, mode=workloads.SOFTMAX_TOPK, seed=53)
    _full_check(w, fused=True)


def test_combine_column_chunks_with_capacity():
    """Rows too long for one ring unit at top-8 (14 KiB: two column chunks
    per row, so units = 2 T and the unit's token a 32-bit division) under a
    capacity (units from both ends of each block's share): every output
    against the oracle."""
    w = workloads.Workload("chunks_cap", T=2001, H=7168, E=16, k=8, P=4, logit_std=1.5, zipf_bias=True,
                           capacity_factor=1.25, seed=54)
    _full_check(w, fused=True)
