"""GPU parity of the re-assigning layout (capacity overflow sent to the
least-loaded expert) against the oracle: every layout array bit-exact, then
dispatch and combine over it."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import workloads
from test_gpu_parity import _full_check

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()
    torch.cuda.init()


def _ra(base, T=None, name=None, **kw):
    w = base if T is None else base.scaled(T)
    return workloads.Workload(**{**w.__dict__, "name": name or (w.name + "_ra"), "reassign": True, **kw})


SMALL = [
    _ra(W["prefill_cap"], 700),
    _ra(W["prefill_cap"], 3001),                      # several layout tiles, ragged tail
    _ra(W["fp8_skewed"], 1500, capacity_factor=1.25),  # k = 2, Zipf-hot experts, FP8 transport
    _ra(W["fine_shared"], 333, capacity_factor=1.25, zipf_bias=True, logit_std=2.0,
        name="fine_shared_ra"),  # softmax-then-top-k, shared experts
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_reassign_small_exact(w):
    plan, L, _ = _full_check(w)
    assert np.any(L["capacity_mask"] == 2), "the case must re-assign something"


def test_reassign_full_size():
    plan, L, _ = _full_check(W["prefill_reassign"])
    assert L["dropped"] == 0 and np.all(L["counts"] <= W["prefill_reassign"].capacity)


def _edge(T, H, E, k, P, cap_factor=1.25, seed=91, **kw):
    return workloads.Workload(f"ra_T{T}_E{E}_k{k}_P{P}", T=T, H=H, E=E, k=k, P=P, capacity_factor=cap_factor,
                              seed=seed, reassign=True, **kw)


EDGES = [
    _edge(257, 64, 256, 16, 256, zipf_bias=True, logit_std=3.0),  # E = P = 256: pairwise partition path
    _edge(900, 32, 8, 1, 2, zipf_bias=True, logit_std=4.0),       # k = 1, heavy overflow
    _edge(4000, 16, 16, 4, 4, zipf_bias=True, logit_std=5.0),     # many tiles, most slots moved
]


@pytest.mark.parametrize("w", EDGES, ids=[w.name for w in EDGES])
def test_reassign_edge_cases(w):
    _full_check(w)
