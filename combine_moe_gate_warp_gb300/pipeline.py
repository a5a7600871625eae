"""One route -> dispatch -> combine pass over the C ABI, with its buffers.

``RoutePlan`` allocates (through PyTorch) every buffer the four calls need
for one problem size and exposes the calls as methods; ``step`` runs the
whole hot path on the current stream.  Each method is a direct call of the
matching C entry point.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import abi


@dataclass
class RouteShape:
    T: int
    H: int
    E: int
    k: int
    P: int
    mode: int = abi.MOE_TOPK_SOFTMAX
    fp8: bool = False
    Ks: int = 0
    capacity: int = 0


class RoutePlan:
    def __init__(self, shape: RouteShape, device="cuda", stream=None):
        s = self.shape = shape
        self.device = torch.device(device)
        self.stream = stream
        T, E, k = s.T, s.E, s.k
        i32 = dict(dtype=torch.int32, device=self.device)
        self.topk_idx = torch.empty((max(T, 1), k), **i32)
        self.gates = torch.empty((max(T, 1), k), dtype=torch.float32, device=self.device)
        self.expert_counts = torch.empty(E, **i32)
        self.aux_loss = torch.empty(1, dtype=torch.float64, device=self.device)
        self.entropy = torch.empty(1, dtype=torch.float64, device=self.device)
        self.ws = abi.alloc_workspace(T, E, k, s.P, self.device, stream)
        self.layout = abi.Layout(T, E, k, s.P, s.capacity, self.device)
        self.r_max = self.layout.r_max
        rows = max(self.r_max, 1)
        if s.fp8:
            self.packed = torch.empty((rows, s.H), dtype=torch.uint8, device=self.device)
            self.scales = torch.empty((rows, 2), dtype=torch.float32, device=self.device)
        else:
            self.packed = torch.empty((rows, s.H), dtype=torch.bfloat16, device=self.device)
            self.scales = None
        self.y = torch.empty((max(T, 1), s.H), dtype=torch.bfloat16, device=self.device)

    # the four hot-path calls -------------------------------------------------
    def gate(self, logits: torch.Tensor):
        s = self.shape
        abi.moe_gate(logits, s.k, s.mode, self.topk_idx, self.gates, self.expert_counts,
                     self.aux_loss, self.entropy, self.ws, self.stream)

    def dispatch_layout(self):
        s = self.shape
        abi.moe_dispatch_layout(self.topk_idx, self.expert_counts, s.T, s.E, s.k, s.P, s.capacity,
                                self.gates, self.layout, self.ws, self.stream)

    def dispatch(self, x: torch.Tensor):
        s = self.shape
        abi.moe_dispatch(x, s.T, s.H, self.layout, int(s.fp8), self.packed, self.scales, self.stream)

    def combine(self, expert_out: torch.Tensor, shared_out: torch.Tensor | None = None):
        s = self.shape
        abi.moe_combine(expert_out, self.layout, self.gates, shared_out, s.Ks, s.T, s.H, self.y,
                        self.stream)

    def step(self, logits, x, expert_out, shared_out=None):
        """gate -> layout -> dispatch -> combine (4 kernel launches)."""
        self.gate(logits)
        self.dispatch_layout()
        self.dispatch(x)
        self.combine(expert_out, shared_out)

    KERNELS_PER_STEP = 4

    def status(self) -> int:
        return abi.moe_get_status(self.ws, self.stream)
