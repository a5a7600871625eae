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
    fp8: int = 0          # dispatch transport: 0 bf16, else a MOE_FP8_* quantiser mode
    Ks: int = 0
    capacity: int = 0
    fp8_combine: int = 0  # expert outputs: 0 bf16, else quantised with this MOE_FP8_* mode


def _check_input(t, dtype, shape, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}")
    if tuple(t.shape[:len(shape)]) != tuple(shape):
        raise ValueError(f"{name}: expected leading shape {tuple(shape)}, got {tuple(t.shape)}")


class RoutePlan:
    """Buffers and bound arguments of one problem size.  The plan is bound to
    ``stream`` (default: the stream current when it is built); its methods
    call the C entry points with cached pointers, so the per-call host cost
    is one foreign call plus input checks."""

    def __init__(self, shape: RouteShape, device="cuda", stream=None):
        s = self.shape = shape
        self.device = torch.device(device)
        self.stream = torch.cuda.current_stream(self.device) if stream is None else stream
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
        if s.fp8_combine:
            self.eo_codes = torch.empty((rows, s.H), dtype=torch.uint8, device=self.device)
            self.eo_scales = torch.empty((rows, 2), dtype=torch.float32, device=self.device)
        self._bind()

    def _bind(self):
        import ctypes
        s = self.shape
        self._lib = abi.lib()
        self._s = ctypes.c_void_p(self.stream.cuda_stream)
        self._Lref = ctypes.byref(self.layout.c)
        self._ws_bytes = self.ws.numel()
        self._gate_tail = (self.topk_idx.data_ptr(), self.gates.data_ptr(), self.expert_counts.data_ptr(),
                           self.aux_loss.data_ptr(), self.entropy.data_ptr(), self.ws.data_ptr(),
                           self._ws_bytes, self._s)
        self._layout_args = (self.topk_idx.data_ptr(), self.expert_counts.data_ptr(), s.T, s.E, s.k, s.P,
                             s.capacity, self.gates.data_ptr(), self._Lref, self.ws.data_ptr(),
                             self._ws_bytes, self._s)
        self._scales_ptr = None if self.scales is None else self.scales.data_ptr()

    # the four hot-path calls -------------------------------------------------
    def gate(self, logits: torch.Tensor):
        s = self.shape
        _check_input(logits, torch.float32, (s.T, s.E), "logits")
        abi._check(self._lib.moe_gate(logits.data_ptr(), s.T, s.E, s.k, s.mode, *self._gate_tail), "moe_gate")

    def dispatch_layout(self):
        abi._check(self._lib.moe_dispatch_layout(*self._layout_args), "moe_dispatch_layout")

    def dispatch(self, x: torch.Tensor):
        s = self.shape
        _check_input(x, torch.bfloat16, (s.T, s.H), "x")
        abi._check(self._lib.moe_dispatch(x.data_ptr(), s.T, s.H, self._Lref, int(s.fp8), self.packed.data_ptr(),
                                          self._scales_ptr, self._s), "moe_dispatch")

    def combine(self, expert_out: torch.Tensor, shared_out: torch.Tensor | None = None):
        s = self.shape
        _check_input(expert_out, torch.bfloat16, (), "expert_out")
        if expert_out.shape[-1] != s.H:
            raise ValueError("expert_out: last dimension must be H")
        sh = None
        if s.Ks:
            _check_input(shared_out, torch.bfloat16, (s.Ks, s.T, s.H), "shared_out")
            sh = shared_out.data_ptr()
        abi._check(self._lib.moe_combine(expert_out.data_ptr(), self._Lref, self.gates.data_ptr(), sh, s.Ks, s.T,
                                         s.H, self.y.data_ptr(), self._s), "moe_combine")

    def quantize_expert_out(self, expert_out: torch.Tensor):
        """FP8-encode the expert-output rows (the expert side of the return
        transport) into eo_codes / eo_scales."""
        s = self.shape
        _check_input(expert_out, torch.bfloat16, (), "expert_out")
        if expert_out.shape[-1] != s.H:
            raise ValueError("expert_out: last dimension must be H")
        abi._check(self._lib.moe_quantize_rows(expert_out.data_ptr(), self._Lref, s.H, s.fp8_combine,
                                               self.eo_codes.data_ptr(), self.eo_scales.data_ptr(), self._s),
                   "moe_quantize_rows")

    def combine_fp8(self, shared_out: torch.Tensor | None = None):
        """Combine from eo_codes / eo_scales."""
        s = self.shape
        sh = None
        if s.Ks:
            _check_input(shared_out, torch.bfloat16, (s.Ks, s.T, s.H), "shared_out")
            sh = shared_out.data_ptr()
        abi._check(self._lib.moe_combine_fp8(self.eo_codes.data_ptr(), self.eo_scales.data_ptr(), self._Lref,
                                             self.gates.data_ptr(), sh, s.Ks, s.T, s.H, self.y.data_ptr(), self._s),
                   "moe_combine_fp8")

    def step(self, logits, x, expert_out, shared_out=None):
        """gate -> layout -> dispatch -> combine; with FP8 expert outputs the
        combine is quantise (expert side) -> FP8 combine."""
        self.gate(logits)
        self.dispatch_layout()
        self.dispatch(x)
        if self.shape.fp8_combine:
            self.quantize_expert_out(expert_out)
            self.combine_fp8(shared_out)
        else:
            self.combine(expert_out, shared_out)

    def launches_per_step(self) -> int:
        """Kernel launches of one step (the grouped FP8 modes take two)."""
        s = self.shape
        n = 3 + (2 if s.fp8 in (abi.MOE_FP8_PER_EXPERT, abi.MOE_FP8_GLOBAL) else 1)
        if s.fp8_combine:
            n += 1 + (2 if s.fp8_combine in (abi.MOE_FP8_PER_EXPERT, abi.MOE_FP8_GLOBAL) else 1)
        return n

    # backward through the same layout -------------------------------------
    def _bwd_buffers(self):
        if getattr(self, "d_expert_out", None) is None:
            s = self.shape
            dev = self.device
            self.d_expert_out = torch.empty((max(self.r_max, 1), s.H), dtype=torch.bfloat16, device=dev)
            self.d_gates = torch.empty((max(s.T, 1), s.k), dtype=torch.float32, device=dev)
            self.dx = torch.empty((max(s.T, 1), s.H), dtype=torch.bfloat16, device=dev)
            self.d_logits = torch.empty((max(s.T, 1), s.E), dtype=torch.float32, device=dev)

    def combine_backward(self, dy: torch.Tensor, expert_out: torch.Tensor):
        """d_expert_out (rows of g*dy) and d_gates (<dy, expert row>)."""
        s = self.shape
        self._bwd_buffers()
        _check_input(dy, torch.bfloat16, (s.T, s.H), "dy")
        _check_input(expert_out, torch.bfloat16, (), "expert_out")
        if expert_out.shape[-1] != s.H:
            raise ValueError("expert_out: last dimension must be H")
        abi._check(self._lib.moe_combine_backward(dy.data_ptr(), expert_out.data_ptr(), self._Lref,
                                                  self.gates.data_ptr(), s.T, s.H, self.d_expert_out.data_ptr(),
                                                  self.d_gates.data_ptr(), self._s), "moe_combine_backward")

    def dispatch_backward(self, d_packed: torch.Tensor):
        """dx = sum of the gradients of each token's packed copies (fp32)."""
        s = self.shape
        self._bwd_buffers()
        _check_input(d_packed, torch.bfloat16, (), "d_packed")
        if d_packed.shape[-1] != s.H:
            raise ValueError("d_packed: last dimension must be H")
        abi._check(self._lib.moe_dispatch_backward(d_packed.data_ptr(), self._Lref, s.T, s.H, self.dx.data_ptr(),
                                                   self._s), "moe_dispatch_backward")

    def gate_backward(self, logits: torch.Tensor, d_gates: torch.Tensor | None = None):
        """d_logits from d_gates (default: the combine backward's d_gates)."""
        s = self.shape
        self._bwd_buffers()
        _check_input(logits, torch.float32, (s.T, s.E), "logits")
        dg = self.d_gates[:s.T] if d_gates is None else d_gates
        _check_input(dg, torch.float32, (s.T, s.k), "d_gates")
        abi._check(self._lib.moe_gate_backward(logits.data_ptr(), self.topk_idx.data_ptr(), dg.data_ptr(), s.T, s.E,
                                               s.k, s.mode, self.d_logits.data_ptr(), self.ws.data_ptr(),
                                               self._ws_bytes, self._s), "moe_gate_backward")

    def backward(self, logits, dy, expert_out, d_packed):
        """combine backward -> gate backward, and the dispatch backward of the
        expert-side gradient d_packed (3 kernel launches)."""
        self.combine_backward(dy, expert_out)
        self.gate_backward(logits)
        self.dispatch_backward(d_packed)

    def status(self) -> int:
        return abi.moe_get_status(self.ws, self.stream)
