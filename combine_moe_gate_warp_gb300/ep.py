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
(source, local expert) pair.

De-duplicated exchange (`dispatch_dedup` / `combine_dedup`): the DeepEP
form of sec. 7's dispatch detail, in which everything bound for one
destination is packed together, sends a token to a rank once however many of
that rank's experts it selected, with those experts' rank-local ids and gates
(moe_dedup_layout with one partition per rank).  The receiver expands the rows
to its experts with moe_dispatch_layout (an id of -1 marks an empty slot) and
moe_dispatch, runs the experts, combines each received row's slots with
moe_combine into one partial row and sends the partials back; the source adds
them with moe_combine_partials.

torch.distributed carries the bytes (NCCL between GPUs, gloo on CPU ranks);
no routing arithmetic happens here, only split sizes and count totals.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


def _layout_counts(layout_or_counts):
    """(kept rows per expert [E], rows to allocate for returned rows or
    None).  Accepts a Layout (its `counts` and `r_max`) or the counts
    tensor itself."""
    if isinstance(layout_or_counts, torch.Tensor):
        return layout_or_counts, None
    return layout_or_counts.counts, int(layout_or_counts.r_max)


@dataclass
class DedupReceived:
    """What one rank receives in a de-duplicated dispatch.  Rows are ordered
    by source rank, then in each source's token order."""
    rows: torch.Tensor           # [n, H] bf16 rows, or uint8 e4m3 codes
    slot_local: torch.Tensor     # [n, k] int32 ids of this rank's experts (0 .. E/W-1), -1 = empty slot
    slot_gate: torch.Tensor      # [n, k] fp32 gates of those slots (0 for empty ones)
    scales: torch.Tensor | None  # [n, 2] fp32 (scale, zero) per row for e4m3 rows
    expert_counts: torch.Tensor  # [E/W] int32: slots each local expert receives (moe_dispatch_layout's counts)
    recv_splits: list            # rows received from each source rank
    send_splits: list            # rows this rank sent to each destination rank

    @property
    def n(self) -> int:
        return sum(self.recv_splits)


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
    def exchange_counts(self, layout_counts) -> torch.Tensor:
        """layout_counts: this rank's KEPT rows per expert [E] -- the layout's
        `counts` (moe_layout.counts, after the capacity), not the gate's
        expert_counts (assignments before the capacity); a Layout is accepted
        too.  Returns [W, E/W] int64 (host): rows that each source rank sends
        to each of this rank's experts."""
        counts, _ = _layout_counts(layout_counts)
        if counts.numel() != self.E:
            raise ValueError(f"layout_counts has {counts.numel()} entries, expected E = {self.E}")
        send = counts.to(torch.int64).reshape(self.W, self.local_experts).contiguous()
        recv = torch.empty_like(send)
        dist.all_to_all_single(recv, send, group=self.group)
        return recv.cpu()

    def _send_splits(self, counts: torch.Tensor) -> list[int]:
        return counts.to(torch.int64).cpu().reshape(self.W, self.local_experts).sum(1).tolist()

    # -- dispatch ----------------------------------------------------------------
    def dispatch(self, packed: torch.Tensor, layout_counts, scales: torch.Tensor | None = None):
        """Send each rank its slice of the packed rows (and of the per-row
        FP8 scales, if given).  `layout_counts`: the layout's kept rows per
        expert (moe_layout.counts) or the Layout itself.  Returns (received
        rows, received scales or None, recv_counts [W, E/W])."""
        counts, _ = _layout_counts(layout_counts)
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
    def combine(self, expert_out_recv: torch.Tensor, recv_counts: torch.Tensor, layout_counts,
                out: torch.Tensor | None = None) -> torch.Tensor:
        """Return every expert-output row to its source: rows [0, R) of the
        result are this rank's expert outputs in its own packed-row order,
        ready for moe_combine with its own layout.  Given the Layout (not
        just its counts) the result is allocated with the layout's r_max rows,
        the size moe_combine requires; rows [R, r_max) are left unwritten."""
        counts, rows = _layout_counts(layout_counts)
        back_send = recv_counts.sum(1).tolist()
        back_recv = self._send_splits(counts)
        R = sum(back_recv)
        if expert_out_recv.shape[0] != sum(back_send):
            raise ValueError(f"{expert_out_recv.shape[0]} expert-output rows for {sum(back_send)} received rows")
        if out is None:
            n = max(R, rows or 0, 1)
            out = expert_out_recv.new_empty((n,) + tuple(expert_out_recv.shape[1:]))
        elif out.shape[0] < R:
            raise ValueError(f"out holds {out.shape[0]} rows, {R} come back")
        dist.all_to_all_single(out[:R], expert_out_recv.contiguous(), back_recv, back_send, group=self.group)
        return out

    # -- de-duplicated send rows -----------------------------------------------
    def dispatch_dedup(self, send_buf: torch.Tensor, send_offsets: torch.Tensor, slot_local: torch.Tensor,
                       slot_gate: torch.Tensor, layout_counts, scales: torch.Tensor | None = None) -> DedupReceived:
        """Send each rank the rows bound for it once per token.

        send_buf [>= S, H], slot_local / slot_gate [>= S, k], scales [>= S, 2]
        or None: the send rows of moe_dedup_layout / moe_dispatch_dedup made
        with one partition per rank (W groups of E/W experts), so that
        send_offsets [W+1] delimits the rows for each destination rank and
        slot_local holds ids of the destination's experts.  layout_counts: the
        layout's kept rows per expert (or the Layout), from which each
        receiver learns how many slots each of its experts receives."""
        counts, _ = _layout_counts(layout_counts)
        offs = [int(v) for v in send_offsets.to(torch.int64).cpu().tolist()]
        if len(offs) != self.W + 1 or offs[0] != 0 or any(b < a for a, b in zip(offs, offs[1:])):
            raise ValueError(f"send_offsets must be the W + 1 = {self.W + 1} row offsets of one partition per rank")
        S = offs[-1]
        k = slot_local.shape[1] if slot_local.dim() == 2 else 0
        for t, name in ((send_buf, "send_buf"), (slot_local, "slot_local"), (slot_gate, "slot_gate"),
                        (scales, "scales")):
            if t is not None and t.shape[0] < S:
                # refuse before any collective, as dispatch() does
                raise ValueError(f"{name} holds {t.shape[0]} rows, send_offsets send {S}")
        if slot_gate.shape[1:] != slot_local.shape[1:]:
            raise ValueError("slot_local and slot_gate must have the same shape")
        send_splits = [offs[i + 1] - offs[i] for i in range(self.W)]
        recv_counts = self.exchange_counts(counts)
        split_t = torch.tensor(send_splits, dtype=torch.int64, device=counts.device)
        recv_t = torch.empty_like(split_t)
        dist.all_to_all_single(recv_t, split_t, group=self.group)
        recv_splits = [int(v) for v in recv_t.cpu().tolist()]
        n = sum(recv_splits)

        def move(t):
            r = t.new_empty((n,) + tuple(t.shape[1:]))
            dist.all_to_all_single(r, t[:S].contiguous(), recv_splits, send_splits, group=self.group)
            return r

        rows = move(send_buf)
        ids = move(slot_local)
        gts = move(slot_gate)
        sc = move(scales) if scales is not None else None
        expert_counts = recv_counts.sum(0).to(torch.int32).to(send_buf.device)
        assert ids.shape[1:] == (k,)
        return DedupReceived(rows=rows, slot_local=ids, slot_gate=gts, scales=sc, expert_counts=expert_counts,
                             recv_splits=recv_splits, send_splits=send_splits)

    def combine_dedup(self, partials_recv: torch.Tensor, received: DedupReceived,
                      out: torch.Tensor | None = None, rows: int | None = None) -> torch.Tensor:
        """Return one partial row per received send row to its source:
        rows [0, S) of the result are this rank's partials in its own
        send-row order, ready for moe_combine_partials.  The result holds
        max(S, rows) rows (pass the moe_dedup's s_max)."""
        S = sum(received.send_splits)
        if partials_recv.shape[0] < received.n:
            raise ValueError(f"{partials_recv.shape[0]} partial rows for {received.n} received rows")
        if out is None:
            out = partials_recv.new_empty((max(S, rows or 0, 1),) + tuple(partials_recv.shape[1:]))
        elif out.shape[0] < S:
            raise ValueError(f"out holds {out.shape[0]} rows, {S} come back")
        dist.all_to_all_single(out[:S], partials_recv[:received.n].contiguous(), received.send_splits,
                               received.recv_splits, group=self.group)
        return out


__all__ = ["ExpertParallelExchange", "DedupReceived"]
