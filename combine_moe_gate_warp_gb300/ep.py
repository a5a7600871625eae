"""Expert-parallel exchange of the packed partitions.

"MoE data traits ... DeepEP and MoE all-to-all data handling" sec. 7: every
rank routes its own tokens, packs the rows bound for the experts of rank j
into one contiguous block and sends it to rank j (dispatch all-to-all); the
experts run on the rows they received; the inverse exchange returns every
output row to its source (combine all-to-all), where moe_combine places it
with the source's own saved indices (sec. 7.5.2, no second routing).  The
exact row counts are known before any data moves (sec. 8.3.A): they are
exchanged first, at expert granularity, so a receiver can size its buffer
and knows where each of its experts' rows start.

Layout convention: partition p of a moe_layout holds experts
[p*E/P, (p+1)*E/P) as one contiguous slice of the packed rows, and rank r of
a world of W ranks owns partitions [r*P/W, (r+1)*P/W) (P % W == 0), i.e.
experts [r*E/W, (r+1)*E/W).  The packed buffer is therefore already ordered
by destination rank: the dispatch exchange is a single all_to_all_single
with split sizes taken from the layout's per-expert counts.

Received rows are ordered by source rank, then by expert within the source,
then in the source's token order; `segments()` gives the row range of each
(source, local expert) pair.  torch.distributed carries the bytes (NCCL
between GPUs, gloo on CPU ranks); no routing arithmetic happens here.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class ExpertParallelExchange:
    """The two all-to-all exchanges of expert parallelism for one layout
    shape (E experts in P partitions over the ranks of `group`)."""

    def __init__(self, E: int, P: int, group=None):
        self.group = group
        self.W = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if P % self.W != 0 or E % P != 0:
            raise ValueError("partitions must divide evenly over the ranks and the experts over the partitions")
        self.E, self.P = E, P
        self.local_experts = E // self.W

    # -- counts ------------------------------------------------------------------
    def exchange_counts(self, counts: torch.Tensor) -> torch.Tensor:
        """counts: this rank's rows per expert [E].  Returns [W, E/W] int64
        (host): rows that each source rank sends to each of this rank's
        experts."""
        send = counts.to(torch.int64).reshape(self.W, self.local_experts).contiguous()
        recv = torch.empty_like(send)
        dist.all_to_all_single(recv, send, group=self.group)
        return recv.cpu()

    def _send_splits(self, counts: torch.Tensor) -> list[int]:
        return counts.to(torch.int64).cpu().reshape(self.W, self.local_experts).sum(1).tolist()

    # -- dispatch ----------------------------------------------------------------
    def dispatch(self, packed: torch.Tensor, counts: torch.Tensor, scales: torch.Tensor | None = None):
        """Send each rank its slice of the packed rows (and of the per-row
        FP8 scales, if given).  Returns (received rows, received scales or
        None, recv_counts [W, E/W])."""
        send_splits = self._send_splits(counts)
        R = sum(send_splits)
        if packed.shape[0] < R or (scales is not None and scales.shape[0] < R):
            # refuse before any collective: the peers see this rank fail
            # (the process group's timeout ends their pending exchange)
            raise ValueError(f"packed buffer holds {packed.shape[0]} rows, the counts send {R}")
        recv_counts = self.exchange_counts(counts)
        recv_splits = recv_counts.sum(1).tolist()
        recv = packed.new_empty((sum(recv_splits),) + tuple(packed.shape[1:]))
        dist.all_to_all_single(recv, packed[:R].contiguous(), recv_splits, send_splits, group=self.group)
        recv_scales = None
        if scales is not None:
            recv_scales = scales.new_empty((sum(recv_splits),) + tuple(scales.shape[1:]))
            dist.all_to_all_single(recv_scales, scales[:R].contiguous(), recv_splits, send_splits, group=self.group)
        return recv, recv_scales, recv_counts

    def segments(self, recv_counts: torch.Tensor) -> list[tuple[int, int, int, int]]:
        """(source rank, global expert, first row, end row) of every received
        segment, in buffer order."""
        out = []
        row = 0
        for src in range(self.W):
            for el in range(self.local_experts):
                n = int(recv_counts[src, el])
                out.append((src, self.rank * self.local_experts + el, row, row + n))
                row += n
        return out

    # -- combine -----------------------------------------------------------------
    def combine(self, expert_out_recv: torch.Tensor, recv_counts: torch.Tensor, counts: torch.Tensor,
                out: torch.Tensor | None = None) -> torch.Tensor:
        """Return every expert-output row to its source: the result is this
        rank's expert outputs in its own packed-row order ([R, ...]), ready
        for moe_combine with its own layout."""
        back_send = recv_counts.sum(1).tolist()
        back_recv = self._send_splits(counts)
        R = sum(back_recv)
        if expert_out_recv.shape[0] != sum(back_send):
            raise ValueError(f"{expert_out_recv.shape[0]} expert-output rows for {sum(back_send)} received rows")
        if out is None:
            out = expert_out_recv.new_empty((R,) + tuple(expert_out_recv.shape[1:]))
        dist.all_to_all_single(out[:R], expert_out_recv.contiguous(), back_recv, back_send, group=self.group)
        return out


__all__ = ["ExpertParallelExchange"]
