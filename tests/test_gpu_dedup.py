"""GPU parity of the per-partition de-duplicated path against the oracle,
stage by stage: the send rows (moe_dedup_layout), the once-per-partition
copies (moe_dispatch_dedup, bf16 and per-token FP8), each partition's
expansion (moe_dispatch_layout with empty slots + moe_dispatch), its partial
combine (moe_combine), and the source's sum of the partials
(moe_combine_partials, with shared experts).  Every stage bit-exact; the
oracle is fed its own outputs and the seeded inputs only."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_gate_warp_gb300 import RoutePlan, abi, workloads
from gpu_util import bits, check_layout, gate_with_oracle, shape_of

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import combine_moe_gate_warp_gb300 as pkg
    pkg.build()
    oracle.build()
    torch.cuda.init()


def _expert_np(e, rows_bits):
    f = (rows_bits.astype(np.uint32) << 16).view(np.float32) * np.float32((e + 1) / 8.0)
    u = f.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _expert_gpu(e, rows):
    return (rows.float() * ((e + 1) / 8.0)).to(torch.bfloat16)


def _check(w, fp8=0):
    T, k, P, E, H = w.T, w.k, w.P, w.E, w.H
    per = E // P
    inp = workloads.make_inputs(w, "cuda")
    plan = RoutePlan(shape_of(w), "cuda")
    _, og = gate_with_oracle(w, plan, inp["logits"])
    plan.dispatch_layout()
    assert plan.status() == 0
    L = check_layout(w, plan, og)
    # send rows
    D = abi.Dedup(T, k, P, "cuda")
    abi.moe_dedup_layout(plan.layout, plan.gates, D)
    Do = oracle.dedup_layout(L["dst_row"], L["offsets"], L["gates"], T, E, k, P)
    S = Do["S"]
    assert plan.status() == 0
    assert np.array_equal(D.send_offsets.cpu().numpy(), Do["send_offsets"])
    assert np.array_equal(D.send_row.cpu().numpy()[:T], Do["send_row"])
    assert np.array_equal(D.send_token.cpu().numpy()[:S], Do["send_token"])
    assert np.array_equal(D.slot_local.cpu().numpy()[:S], Do["slot_local"])
    assert np.array_equal(D.slot_gate.cpu().numpy()[:S].view(np.uint32), Do["slot_gate"].view(np.uint32))
    # copies, once per (token, partition)
    x_bits = bits(inp["x"])
    if fp8:
        send = torch.empty((D.s_max, H), dtype=torch.uint8, device="cuda")
        sc = torch.empty((D.s_max, 2), dtype=torch.float32, device="cuda")
        abi.moe_dispatch_dedup(inp["x"], T, H, D, 1, send, sc)
        want, want_s = oracle.quantize_rows_grouped(x_bits, Do["send_token"].astype(np.int64),
                                                    np.arange(S, dtype=np.int32), S)
        assert np.array_equal(send[:S].cpu().numpy(), want)
        assert np.array_equal(sc[:S].cpu().numpy().view(np.uint32), want_s.view(np.uint32))
        return
    send = torch.empty((D.s_max, H), dtype=torch.bfloat16, device="cuda")
    abi.moe_dispatch_dedup(inp["x"], T, H, D, 0, send)
    assert np.array_equal(bits(send[:S]), x_bits[Do["send_token"]])
    # each partition: expand, experts, partial combine
    partials = torch.empty((D.s_max, H), dtype=torch.bfloat16, device="cuda")
    partials_o = np.zeros((max(S, 1), H), np.uint16)
    offs = Do["send_offsets"]
    for p in range(P):
        s0, s1 = int(offs[p]), int(offs[p + 1])
        n = s1 - s0
        if n == 0:
            continue
        lw = workloads.Workload(f"recv{p}", T=n, H=H, E=per, k=k, P=1)
        rp = RoutePlan(shape_of(lw), "cuda")
        rp.topk_idx[:n].copy_(D.slot_local[s0:s1])
        rp.gates[:n].copy_(D.slot_gate[s0:s1])
        rp.expert_counts.copy_(plan.layout.counts[p * per:(p + 1) * per])
        rp.dispatch_layout()
        rp.dispatch(send[s0:s1])
        Lo = oracle.layout(Do["slot_local"][s0:s1], per, 1, 0, gates_f32=Do["slot_gate"][s0:s1])
        assert np.array_equal(rp.layout.dst_row.cpu().numpy()[:n * k], Lo["dst_row"])
        assert np.array_equal(rp.layout.offsets.cpu().numpy(), Lo["offsets"])
        Rl = Lo["R"]
        eo = torch.empty((max(rp.r_max, 1), H), dtype=torch.bfloat16, device="cuda")
        local_o = oracle.dispatch_bf16_rows(x_bits[Do["send_token"][s0:s1]], k, Lo["src_pos"], np.arange(Rl))
        eo_o = np.empty_like(local_o)
        for el in range(per):
            a0, a1 = int(Lo["offsets"][el]), int(Lo["offsets"][el + 1])
            eo[a0:a1] = _expert_gpu(p * per + el, rp.packed[a0:a1])
            eo_o[a0:a1] = _expert_np(p * per + el, local_o[a0:a1])
        rp.combine(eo)
        assert rp.status() == 0
        partials[s0:s1] = rp.y[:n]
        partials_o[s0:s1] = oracle.combine_f32order(eo_o if Rl else np.zeros((1, H), np.uint16), Lo["gates"],
                                                    Lo["dst_row"], np.arange(n), n, k)
    assert np.array_equal(bits(partials[:S]), partials_o[:S])
    # the source adds the partials (+ shared experts)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    abi.moe_combine_partials(partials, D, inp["shared"], w.Ks, T, H, y)
    assert plan.status() == 0
    sh = None if inp["shared"] is None else bits(inp["shared"])
    y_o = oracle.combine_f32order(partials_o, np.ones((T, P), np.float32), Do["send_row"].ravel(), np.arange(T), T, P,
                                  sh)
    assert np.array_equal(bits(y), y_o)


@pytest.mark.parametrize("w", [W["v2_top2"].scaled(1500), W["fine_shared"].scaled(700),
                               W["prefill_cap"].scaled(1200), W["prefill_reassign"].scaled(900)],
                         ids=lambda w: w.name)
def test_dedup_path_bf16(w):
    _check(w)


def test_dedup_dispatch_fp8():
    _check(W["fp8_skewed"].scaled(1000), fp8=1)


def test_dedup_large():
    # prefill_cap's shape (k = 8 over 8 partitions, H = 4096) at 16384 tokens: 8 tiles of the
    # send-row kernels, ~100 K send rows
    _check(W["prefill_cap"].scaled(16384))
