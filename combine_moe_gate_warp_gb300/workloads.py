"""Seeded synthetic workloads for MoE token routing.

This module only draws random inputs and names the workload shapes; it holds
none of the routing arithmetic.  Both the CUDA path's tests/benchmark and
the CPU oracle receive the *same* tensors from here.

Workloads (shapes taken from the workloads the source pages discuss):

  tiny        T=256,    H=512,  E=8,  k=2, P=4, top-k-then-softmax gates,
              expert outputs = the packed rows themselves (identity experts)
  v2_top2     T=16384 (batch 32 x seq 512), H=5120, E=16, k=2, P=4,
              top-k-then-softmax; the sync-tax guide's batch 32 / seq 512 /
              hidden 5120 example with DeepSeek-V2's 16 experts, top-2
  fine_shared T=8192, H=2048, E=32, k=8, P=8, softmax-over-all-then-top-k
              (no renormalisation), 2 shared experts added in the combine
              (DeepSeekMoE fine-grained experts mN=32, mK=8, K_s=2)
  fp8_skewed  T=65536 (batch 64 x seq 1024), H=4096, E=64, k=2, P=8,
              logits N(0,1) + per-expert bias 2*ln(1/rank_e) (Zipf-like hot
              experts, ranks permuted by the seed); per-token affine FP8 e4m3
              transport
  prefill_cap T=262144 (batch 128 x seq 2048), H=4096, E=64, k=8, P=8,
              logits N(0, 1.5^2) + the same Zipf-like bias, capacity
              ceil(1.25*T*k/E) per expert, bf16 transport
  prefill_reassign
              prefill_cap with the capacity overflow re-assigned to the
              least-loaded expert instead of dropped
  fp8_expert, fp8_global, fp8_both
              fp8_skewed's shape and inputs with per-expert / global FP8
              groups for the dispatch, or per-token FP8 both ways (the
              expert outputs quantised per row and combined from FP8)

Distributions: x ~ N(0,1) drawn in fp32 and rounded to bf16; router logits
fp32 as above; expert outputs (the FFN is not part of this path) and shared
expert outputs ~ N(0,1) rounded to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

TOPK_SOFTMAX = 0
SOFTMAX_TOPK = 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    P: int
    mode: int = TOPK_SOFTMAX
    fp8: int = 0           # dispatch: 0 bf16, 1 per-token, 2 per-expert, 3 global FP8
    Ks: int = 0
    logit_std: float = 1.0
    zipf_bias: bool = False
    capacity_factor: float = 0.0  # 0: no capacity limit
    identity_experts: bool = False
    fp8_combine: int = 0   # expert outputs: 0 bf16, else FP8 with this quantiser mode
    reassign: bool = False  # capacity overflow re-assigned to the least-loaded expert
    seed: int = 1234
    note: str = field(default="", compare=False)

    @property
    def capacity(self) -> int:
        """ceil(factor * T * k / E) in exact integer arithmetic (factor 1.25
        is 5/4); 0 means no limit."""
        if self.capacity_factor <= 0:
            return 0
        assert self.capacity_factor == 1.25, "only the 1.25 factor is defined"
        return (5 * self.T * self.k + 4 * self.E - 1) // (4 * self.E)

    @property
    def r_max(self) -> int:
        A = self.T * self.k
        return A if self.capacity == 0 else min(A, self.E * self.capacity)

    def scaled(self, T: int, name: str | None = None) -> "Workload":
        """Same workload with a different token count (small parity cases)."""
        d = dict(self.__dict__)
        d["T"] = T
        d["name"] = name or f"{self.name}_T{T}"
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=512, E=8, k=2, P=4, identity_experts=True, seed=1234),
    "v2_top2": Workload("v2_top2", T=16384, H=5120, E=16, k=2, P=4, seed=1235),
    "fine_shared": Workload("fine_shared", T=8192, H=2048, E=32, k=8, P=8, mode=SOFTMAX_TOPK,
                            Ks=2, seed=1236),
    "fp8_skewed": Workload("fp8_skewed", T=65536, H=4096, E=64, k=2, P=8, fp8=1,
                           zipf_bias=True, seed=1237),
    "prefill_cap": Workload("prefill_cap", T=262144, H=4096, E=64, k=8, P=8, logit_std=1.5,
                            zipf_bias=True, capacity_factor=1.25, seed=1238),
}
# The other quantiser modes on the fp8_skewed shape and inputs (same seed):
# per-expert and global groups for the dispatch, and FP8 both ways (per-token
# dispatch, per-token expert outputs into an FP8 combine).
for _name, _kw in (("fp8_expert", dict(fp8=2)), ("fp8_global", dict(fp8=3)),
                   ("fp8_both", dict(fp8=1, fp8_combine=1))):
    WORKLOADS[_name] = Workload(**{**WORKLOADS["fp8_skewed"].__dict__, "name": _name, **_kw})
# prefill_cap with the capacity overflow re-assigned instead of dropped
WORKLOADS["prefill_reassign"] = Workload(**{**WORKLOADS["prefill_cap"].__dict__, "name": "prefill_reassign",
                                            "reassign": True})
ORDER = ["tiny", "v2_top2", "fine_shared", "fp8_skewed", "prefill_cap", "fp8_expert", "fp8_global", "fp8_both",
         "prefill_reassign"]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(rows: int, cols: int, g: torch.Generator, device, chunk_elems: int = 1 << 28):
    """N(0,1) drawn in fp32 then rounded to bf16, generated in row chunks so
    the fp32 temporary stays small."""
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    step = max(1, chunk_elems // max(cols, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = torch.randn((r1 - r0, cols), generator=g, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
    return out


def zipf_bias(E: int, seed: int) -> torch.Tensor:
    """Per-expert logit bias 2*ln(1/rank_e), ranks 1..E permuted by the seed
    (CPU generator so the permutation does not depend on the device)."""
    g = _gen("cpu", seed ^ 0x5EED)
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (2.0 * torch.log(1.0 / rank)).to(torch.float32)


def make_logits(w: Workload, device="cuda") -> torch.Tensor:
    g = _gen(device, w.seed)
    logits = torch.randn((w.T, w.E), generator=g, device=device, dtype=torch.float32)
    if w.logit_std != 1.0:
        logits = logits * w.logit_std
    if w.zipf_bias:
        logits = logits + zipf_bias(w.E, w.seed).to(device)
    return logits.contiguous()


def make_x(w: Workload, device="cuda") -> torch.Tensor:
    return _randn_bf16(w.T, w.H, _gen(device, w.seed + 101), device)


def make_shared(w: Workload, device="cuda"):
    if w.Ks == 0:
        return None
    return _randn_bf16(w.Ks * w.T, w.H, _gen(device, w.seed + 202), device).view(w.Ks, w.T, w.H)


def make_expert_out(w: Workload, rows: int, device="cuda") -> torch.Tensor:
    """Seeded stand-in for the expert FFN outputs, in packed-row layout."""
    return _randn_bf16(rows, w.H, _gen(device, w.seed + 303), device)


def make_dy(w: Workload, device="cuda") -> torch.Tensor:
    """Seeded stand-in for the gradient of the combine output y."""
    return _randn_bf16(w.T, w.H, _gen(device, w.seed + 404), device)


def make_d_packed(w: Workload, rows: int, device="cuda") -> torch.Tensor:
    """Seeded stand-in for the gradient of the packed rows (what the expert
    FFN's backward hands to the dispatch backward)."""
    return _randn_bf16(rows, w.H, _gen(device, w.seed + 505), device)


def make_d_gates(w: Workload, device="cuda") -> torch.Tensor:
    """Seeded stand-in for the gradient of the gate weights [T, k] fp32."""
    return torch.randn((w.T, w.k), generator=_gen(device, w.seed + 606), device=device, dtype=torch.float32)


def make_inputs(w: Workload, device="cuda") -> dict:
    return dict(logits=make_logits(w, device), x=make_x(w, device), shared=make_shared(w, device))


def nbytes_roofline(w: Workload, R: int) -> int:
    """Roofline bytes of one route+dispatch+combine pass: x read, packed
    written, expert outputs read, y written."""
    bt = 1 if w.fp8 else 2
    return w.T * w.H * 2 + R * w.H * bt + R * w.H * 2 + w.T * w.H * 2


def nbytes_backward(w: Workload, R: int) -> dict:
    """Roofline bytes of each backward call: combine backward reads dy and
    the kept expert rows and writes their gradients (+ the gate gradients);
    dispatch backward reads the kept row gradients and writes dx; gate
    backward reads the logits and writes their gradients (+ ids, d_gates)."""
    return {
        "combine_backward": w.T * w.H * 2 + 2 * R * w.H * 2 + w.T * w.k * 4 * 3,
        "dispatch_backward": R * w.H * 2 + w.T * w.H * 2 + w.T * w.k * 4,
        "gate_backward": 2 * w.T * w.E * 4 + w.T * w.k * 8,
    }


def gib(n: int) -> float:
    return n / float(1 << 30)


def describe(w: Workload) -> str:
    c = w.capacity
    return (f"{w.name}: T={w.T} H={w.H} E={w.E} k={w.k} P={w.P} mode={w.mode} fp8={int(w.fp8)} "
            f"fp8_combine={w.fp8_combine} "
            f"Ks={w.Ks} capacity={c if c else 'none'}")


__all__ = ["Workload", "WORKLOADS", "ORDER", "make_inputs", "make_logits", "make_x",
           "make_shared", "make_expert_out", "make_dy", "make_d_packed", "make_d_gates", "zipf_bias", "nbytes_roofline",
           "nbytes_backward", "describe",
           "TOPK_SOFTMAX", "SOFTMAX_TOPK", "gib", "math"]
