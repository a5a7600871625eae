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
    reassign: bool = False  # capacity overflow re-assigned to the least-loaded expert (not dropped)


def _check_input(t, dtype, shape, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}")
    if tuple(t.shape[:len(shape)]) != tuple(shape):
        raise ValueError(f"{name}: expected leading shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_packed_rows(t, dtype, r_max, H, name):
    """A tensor in packed-row order: the kernels read it up to the layout's
    row count R, which only the device knows, so it must hold r_max >= R
    rows of H values."""
    if t.dim() != 2 or t.shape[1] != H:
        raise ValueError(f"{name}: expected [rows, {H}], got {tuple(t.shape)}")
    if t.shape[0] < r_max:
        raise ValueError(f"{name}: {t.shape[0]} rows, the layout may hold up to r_max = {r_max}")
    _check_input(t, dtype, (), name)


class RoutePlan:
    """Buffers and bound arguments of one problem size.  The plan is bound to
    ``stream`` (default: the stream current when it is built); its methods
    call the C entry points with cached pointers, so the per-call host cost
    is one foreign call plus input checks."""

    def __init__(self, shape: RouteShape, device="cuda", stream=None, route_stream=None):
        s = self.shape = shape
        self.device = torch.device(device)
        self.stream = torch.cuda.current_stream(self.device) if stream is None else stream
        # gate and layout may run on their own stream (see RoutePipeline)
        self.route_stream = self.stream if route_stream is None else route_stream
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
        self._sr = ctypes.c_void_p(self.route_stream.cuda_stream)
        self._Lref = ctypes.byref(self.layout.c)
        self._ws_bytes = self.ws.numel()
        self._gate_tail = (self.topk_idx.data_ptr(), self.gates.data_ptr(), self.expert_counts.data_ptr(),
                           self.aux_loss.data_ptr(), self.entropy.data_ptr(), self.ws.data_ptr(),
                           self._ws_bytes, self._sr)
        self._layout_args = (self.topk_idx.data_ptr(), self.expert_counts.data_ptr(), s.T, s.E, s.k, s.P,
                             s.capacity, self.gates.data_ptr(), self._Lref, self.ws.data_ptr(),
                             self._ws_bytes, self._sr)
        self._route_tail = (s.T, s.E, s.k, s.mode, s.P, s.capacity, self.topk_idx.data_ptr(), self.gates.data_ptr(),
                            self.expert_counts.data_ptr(), self.aux_loss.data_ptr(), self.entropy.data_ptr(),
                            self._Lref, self.ws.data_ptr(), self._ws_bytes, self._sr)
        # moe_route (gate + layout, one launch where the batch allows) unless
        # the overflow is re-assigned
        self.fused_route = not s.reassign
        self._scales_ptr = None if self.scales is None else self.scales.data_ptr()

    # the four hot-path calls -------------------------------------------------
    def gate(self, logits: torch.Tensor):
        s = self.shape
        _check_input(logits, torch.float32, (s.T, s.E), "logits")
        abi._check(self._lib.moe_gate(logits.data_ptr(), s.T, s.E, s.k, s.mode, *self._gate_tail), "moe_gate")

    def route(self, logits: torch.Tensor):
        """The routing of one batch: moe_route, or moe_gate and then the
        layout call when the capacity overflow is re-assigned."""
        s = self.shape
        if self.fused_route:
            _check_input(logits, torch.float32, (s.T, s.E), "logits")
            abi._check(self._lib.moe_route(logits.data_ptr(), *self._route_tail), "moe_route")
            return
        self.gate(logits)
        self.dispatch_layout()

    def dispatch_layout(self):
        if self.shape.reassign:
            abi._check(self._lib.moe_dispatch_layout_reassign(*self._layout_args), "moe_dispatch_layout_reassign")
        else:
            abi._check(self._lib.moe_dispatch_layout(*self._layout_args), "moe_dispatch_layout")

    def dispatch(self, x: torch.Tensor):
        s = self.shape
        _check_input(x, torch.bfloat16, (s.T, s.H), "x")
        abi._check(self._lib.moe_dispatch(x.data_ptr(), s.T, s.H, self._Lref, int(s.fp8), self.packed.data_ptr(),
                                          self._scales_ptr, self._s), "moe_dispatch")

    def combine(self, expert_out: torch.Tensor, shared_out: torch.Tensor | None = None):
        s = self.shape
        _check_packed_rows(expert_out, torch.bfloat16, self.r_max, s.H, "expert_out")
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
        _check_packed_rows(expert_out, torch.bfloat16, self.r_max, s.H, "expert_out")
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
        """route (gate + layout) -> dispatch -> combine; with FP8 expert
        outputs the combine is quantise (expert side) -> FP8 combine."""
        self.route(logits)
        self.dispatch(x)
        if self.shape.fp8_combine:
            self.quantize_expert_out(expert_out)
            self.combine_fp8(shared_out)
        else:
            self.combine(expert_out, shared_out)

    def launches_per_step(self) -> int:
        """Kernel launches of one step (routing: one, or two when not fused;
        the grouped FP8 modes take two)."""
        s = self.shape
        route = abi.moe_route_launches(s.T, s.E, s.k, s.mode, s.P) if self.fused_route else 2
        n = route + 1 + (2 if s.fp8 in (abi.MOE_FP8_PER_EXPERT, abi.MOE_FP8_GLOBAL) else 1)
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
        _check_packed_rows(expert_out, torch.bfloat16, self.r_max, s.H, "expert_out")
        abi._check(self._lib.moe_combine_backward(dy.data_ptr(), expert_out.data_ptr(), self._Lref,
                                                  self.gates.data_ptr(), s.T, s.H, self.d_expert_out.data_ptr(),
                                                  self.d_gates.data_ptr(), self._s), "moe_combine_backward")

    def dispatch_backward(self, d_packed: torch.Tensor):
        """dx = sum of the gradients of each token's packed copies (fp32)."""
        s = self.shape
        self._bwd_buffers()
        _check_packed_rows(d_packed, torch.bfloat16, self.r_max, s.H, "d_packed")
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
        if self.route_stream is not self.stream:
            self.route_stream.synchronize()
        return abi.moe_get_status(self.ws, self.stream)


class RouteGraph:
    """The one-stream step captured once as a CUDA graph and replayed.

    For small batches the host cost of the step's foreign calls (one per
    kernel) exceeds the kernels' own time; a replay submits every kernel of
    the step in one launch.  The graph reads its inputs from fixed buffers
    (``logits``, ``x``, ``expert_out`` [r_max, H], ``shared_out``) and leaves
    its results in ``plan`` exactly as ``RoutePlan.step`` does; ``step``
    copies new inputs in and replays.  The graph runs on its own stream;
    ``step`` orders it after the caller's current stream and the caller's
    stream after it.  Every kernel runs once before the capture, outside it:
    per-kernel attributes and occupancy are set up on first use, which a
    capture may not do."""

    def __init__(self, shape: RouteShape, device="cuda"):
        self.device = torch.device(device)
        self.stream = torch.cuda.Stream(self.device)
        self.plan = p = RoutePlan(shape, self.device, stream=self.stream)
        s = shape
        bf16 = dict(dtype=torch.bfloat16, device=self.device)
        self.logits = torch.zeros((s.T, s.E), dtype=torch.float32, device=self.device)
        self.x = torch.zeros((s.T, s.H), **bf16)
        self.expert_out = torch.zeros((max(p.r_max, 1), s.H), **bf16)
        self.shared_out = torch.zeros((s.Ks, s.T, s.H), **bf16) if s.Ks else None
        self.graph = None
        if s.T == 0:
            return  # nothing to launch: step() is a no-op
        self.stream.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(self.stream):
            self._calls()
        self.stream.synchronize()
        st = p.status()
        if st != abi.MOE_OK:
            raise abi.MoeError(st, "RouteGraph warm-up")
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._calls()

    def _calls(self):
        self.plan.step(self.logits, self.x, self.expert_out, self.shared_out)

    def replay(self):
        """Replay on the graph's stream (inputs already in the buffers)."""
        if self.graph is None:
            return
        with torch.cuda.stream(self.stream):
            self.graph.replay()

    def step(self, logits=None, x=None, expert_out=None, shared_out=None) -> RoutePlan:
        """Copy the given inputs into the graph's buffers and replay; returns
        the plan holding the results."""
        cur = torch.cuda.current_stream(self.device)
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            for src, dst in ((logits, self.logits), (x, self.x), (shared_out, self.shared_out)):
                if src is not None:
                    dst.copy_(src, non_blocking=True)
            if expert_out is not None:
                self.expert_out[:expert_out.shape[0]].copy_(expert_out, non_blocking=True)
            if self.graph is not None:
                self.graph.replay()
        cur.wait_stream(self.stream)
        return self.plan

    def launches_per_step(self) -> int:
        return self.plan.launches_per_step()

    def status(self) -> int:
        return self.plan.status()


class RoutePipeline:
    """Back-to-back batches with the routing of one overlapping the data
    movement of the previous one ("MoE data traits ... DeepEP and MoE
    all-to-all data handling" sec. 7.5.1 overlap and 7.5.5 double buffering).

    Two plans alternate between batches.  The gate and the layout of batch i
    run on a high-priority routing stream while dispatch and combine of
    batch i-1 run on a data stream: the first two are short chains of
    dependent round trips that leave HBM idle, the last two stream HBM.
    Batch i's dispatch waits for its layout (an event); batch i's gate waits
    until batch i-2, the last user of the same plan, has finished its
    combine.  With two data streams (the default) consecutive batches' data
    calls go to alternate streams, so batch i's dispatch, which needs only
    its own layout, may start while batch i-1's combine still runs instead of
    after it (the two are independent).  Each call is still one C-ABI call;
    nothing is skipped or reordered within a batch.
    """

    def __init__(self, shape: RouteShape, device="cuda", depth: int = 2, route_priority: str = "high",
                 data_streams: int = 2):
        self.device = torch.device(device)
        lo, hi = torch.cuda.Stream.priority_range()
        n = max(1, min(int(data_streams), depth))
        self.data_streams = [torch.cuda.Stream(self.device, priority=lo) for _ in range(n)]
        self.data_stream = self.data_streams[0]
        self.route_stream = torch.cuda.Stream(self.device, priority=hi if route_priority == "high" else lo)
        self.plans = [RoutePlan(shape, self.device, stream=self.data_streams[d % n], route_stream=self.route_stream)
                      for d in range(depth)]
        self._routed = [torch.cuda.Event() for _ in range(depth)]
        self._done = [torch.cuda.Event() for _ in range(depth)]
        self.step_index = 0
        for d, ev in enumerate(self._done):
            ev.record(self.plans[d].stream)

    @staticmethod
    def overlaps(shape: RouteShape) -> bool:
        """Whether back-to-back batches gain from the overlap: every shape the
        path takes.  Measured on GB300: the bf16 workloads run 5-17 % faster
        per batch than on one stream; the FP8 ones, whose encode kernels are
        persistent and fill every SM, gained nothing while the data calls of
        all batches shared one stream, and gain with two alternating data
        streams, where one batch's encode overlaps the previous batch's
        combine (65536 x 4096, top-2, e4m3 dispatch: 422 -> 403 us; FP8 both
        ways: 660 -> 633 us)."""
        return True

    def plan_for(self, i: int) -> RoutePlan:
        return self.plans[i % len(self.plans)]

    def stream_for(self, i: int) -> torch.cuda.Stream:
        """The data stream of step i's dispatch and combine."""
        return self.plan_for(i).stream

    def wait_event(self, ev: torch.cuda.Event):
        """Make every stream of the pipeline wait for `ev`."""
        self.route_stream.wait_event(ev)
        for st in self.data_streams:
            st.wait_event(ev)

    def record(self, ev: torch.cuda.Event):
        """Record `ev` once the work enqueued so far on every data stream is
        done (the first data stream waits for the others)."""
        for st in self.data_streams[1:]:
            self.data_stream.wait_stream(st)
        ev.record(self.data_stream)

    def step(self, logits, x, expert_out, shared_out=None, out=None, stats_out=None) -> RoutePlan:
        """Enqueue one batch; returns the plan whose buffers (y, layout,
        statistics) hold its results once the data stream reaches this
        point, until the plan is reused len(plans) steps later.  With `out`
        ([T, H] bf16, device or pinned host) y is also copied there on the
        data stream, and with `stats_out` ([2] fp64) the aux loss and the
        entropy, before the plan is released.  Inputs must be ready for both
        streams (produced on them, ordered by wait_event, or synchronised)."""
        i = self.step_index
        self.step_index += 1
        d = i % len(self.plans)
        p = self.plans[d]
        self.route_stream.wait_event(self._done[d])
        p.route(logits)
        self._routed[d].record(self.route_stream)
        p.stream.wait_event(self._routed[d])
        p.dispatch(x)
        if p.shape.fp8_combine:
            p.quantize_expert_out(expert_out)
            p.combine_fp8(shared_out)
        else:
            p.combine(expert_out, shared_out)
        if out is not None or stats_out is not None:
            with torch.cuda.stream(p.stream):
                if out is not None:
                    out.copy_(p.y[:p.shape.T], non_blocking=True)
                if stats_out is not None:
                    stats_out[0:1].copy_(p.aux_loss, non_blocking=True)
                    stats_out[1:2].copy_(p.entropy, non_blocking=True)
        self._done[d].record(p.stream)
        return p

    def release_event(self, i: int) -> torch.cuda.Event:
        """Event recorded when step i's plan (and its inputs) were last
        released; a producer of step i's inputs waits on it before
        overwriting buffers that step i-len(plans) read."""
        return self._done[i % len(self.plans)]

    def synchronize(self):
        self.route_stream.synchronize()
        for st in self.data_streams:
            st.synchronize()

    def status(self) -> int:
        """Synchronise and return the first non-zero device status of the plans."""
        self.synchronize()
        for p in self.plans:
            st = p.status()
            if st:
                return st
        return 0

    def launches_per_step(self) -> int:
        return self.plans[0].launches_per_step()
