"""GPU parity of the grouped FP8 quantiser modes (per-expert and global
dispatch, per-token / per-expert / global expert outputs) and of the FP8
combine, against the oracle: codes and scale words bit-exact, the FP8
combine bit-exact in its pinned fp32 order and within its fp64 bound."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import RoutePlan, workloads
from gpu_util import bits, check_combine, check_dispatch, route_checked, shape_of
from test_gpu_parity import _full_check

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()
    torch.cuda.init()


def _variant(base, name, **kw):
    return workloads.Workload(**{**base.__dict__, "name": name, **kw})


SMALL = [
    W["fp8_expert"].scaled(1500),
    W["fp8_global"].scaled(1500),
    W["fp8_both"].scaled(1500),
    _variant(W["fp8_skewed"].scaled(1200), "combine_expert", fp8_combine=2),
    _variant(W["fp8_skewed"].scaled(1200), "combine_global", fp8=3, fp8_combine=3),
    _variant(W["fine_shared"].scaled(333), "shared_fp8_both", fp8=2, fp8_combine=1),   # + shared experts
    _variant(W["prefill_cap"].scaled(700), "capacity_fp8", fp8=2, fp8_combine=2),      # drops
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_fp8_modes_small_exact(w):
    _full_check(w)


@pytest.mark.parametrize("name", ["fp8_expert", "fp8_global", "fp8_both"])
def test_fp8_modes_full_size(name):
    _full_check(W[name])


def _edge(T, H, E, k, P, fp8, fp8c=0, cap=0.0, seed=41, **kw):
    return workloads.Workload(f"fp8m_T{T}_H{H}_E{E}_k{k}_{fp8}{fp8c}", T=T, H=H, E=E, k=k, P=P, fp8=fp8,
                              fp8_combine=fp8c, capacity_factor=cap, seed=seed, **kw)


EDGES = [
    _edge(1, 16, 4, 2, 2, 2, 2),                       # one token, smallest row
    _edge(257, 64, 256, 16, 8, 2, 2),                  # E = 256, k = 16: many groups, empty experts
    _edge(64, 16384, 8, 2, 2, 3, 3),                   # longest rows
    _edge(3000, 32, 16, 4, 4, 2, 3, cap=1.25, zipf_bias=True, logit_std=3.0),  # tokens with no kept slot
    _edge(600, 48, 8, 1, 1, 3, 1),                     # k = 1, ragged 16-column groups
    _edge(333, 80, 8, 2, 4, 1, 1, Ks=2),               # shared experts, 5 groups per row
    _edge(200, 528, 8, 2, 4, 1, 1, Ks=1),              # 33 groups: a full span and a one-group span
]


@pytest.mark.parametrize("w", EDGES, ids=[w.name for w in EDGES])
def test_fp8_modes_edge_cases(w):
    _full_check(w)


def test_constant_groups_and_clean_workspace():
    """All rows of the batch equal: every group is constant (scale 0, zero
    codes).  Then a second, ordinary batch on the same plan: the group keys
    were reset, so it matches the oracle again."""
    w = _edge(500, 64, 8, 2, 4, 3, 2)
    plan = RoutePlan(shape_of(w), "cuda")
    for rep in range(2):
        inp = workloads.make_inputs(workloads.Workload(**{**w.__dict__, "seed": 60 + rep}), "cuda")
        if rep == 0:
            inp["x"][:] = 1.25
        L = route_checked(w, plan, inp["logits"])
        plan.dispatch(inp["x"])
        R = L["R"]
        eo = workloads.make_expert_out(w, max(plan.r_max, 1), "cuda")
        if rep == 0:
            eo[:] = -0.5
        plan.quantize_expert_out(eo)
        plan.combine_fp8(None)
        assert plan.status() == 0
        rows = np.arange(R, dtype=np.int64)
        check_dispatch(w, plan, L, bits(inp["x"]), rows)
        check_combine(w, plan, L, eo, None, np.arange(w.T, dtype=np.int64))
        if rep == 0:
            assert not plan.packed[:R].any() and not plan.eo_codes[:R].any()
            assert torch.all(plan.scales[:R, 0] == 0) and torch.all(plan.scales[:R, 1] == 1.25)
            assert torch.all(plan.y[:w.T].float() == -0.5)


@pytest.mark.parametrize("H,fp8c", [(1024, 1), (2048, 1), (1024, 2)])
def test_expert_rows_split_between_two_warps(H, fp8c):
    """Rows of expert outputs of 1024 columns or more are encoded by two
    warps, each half of the columns, their extremes meeting in shared
    memory.  Rows whose extremes sit in one half only, in the other, and
    signed zeros as extremes (whose sign the ordered keys decide) must give
    the oracle's codes and scales exactly."""
    w = _edge(300, H, 8, 2, 4, 1, fp8c, seed=47)
    plan = RoutePlan(shape_of(w), "cuda")
    inp = workloads.make_inputs(w, "cuda")
    L = route_checked(w, plan, inp["logits"])
    plan.dispatch(inp["x"])
    R = L["R"]
    eo = workloads.make_expert_out(w, max(plan.r_max, 1), "cuda")
    h = H // 2
    eo[0] = 0.0
    eo[0, ::3] = -0.0                      # max +0, min -0: both extremes zero
    eo[1] = -0.0                           # constant -0
    eo[2] = -eo[2].abs()
    eo[2, h:] = -0.0                       # max -0, in the second half only
    eo[3] = eo[3].abs()
    eo[3, 5] = -0.0                        # min -0, in the first half only
    eo[4] = eo[4] * 0.01
    eo[4, H - 1] = 7.0                     # max in the second half,
    eo[4, 0] = -3.0                        # min in the first
    eo[5] = eo[5] * 0.01
    eo[5, h + 1] = 5.0                     # both extremes in the second half
    eo[5, H - 2] = -5.0
    eo[6, :h] = 0.0                        # first half flat zero, second half random
    plan.quantize_expert_out(eo)
    plan.combine_fp8(None)
    assert plan.status() == 0
    check_combine(w, plan, L, eo, None, np.arange(w.T, dtype=np.int64))
    assert R >= 7
