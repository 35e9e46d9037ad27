"""Sharded expert-parallel shuffle: one process (and one GPU) per rank.

The form the pages build the shuffle for ("[Not ready] MSCCLPP EP
implementation", mscclpp pull request 852, section "Scope", Intranode:
get_dispatch_layout on every rank, then intranode_dispatch and
intranode_combine over peer buffers; the internode notify_dispatch commit:
the count exchange that fixes the receiver-side prefix matrices).  Rank s
holds its own T tokens.  dispatch:

  1. layout of the rank's own tokens over R destinations (shard_layout): the
     send buffer is packed destination-major in token order, so the rows for
     destination r are one run;
  2. all-gather of every rank's per-destination counts (and per-expert
     counts): counts[s][r] = tokens of rank s sent to rank r;
  3. offsets from the counts (shard_offsets, host): this rank's runs, and
     where each source's run lands in its receive buffer;
  4. the rank's tokens dispatched into its send buffer (ep_dispatch with the
     send slots), bf16 or FP8 with scales, with the per-row metadata;
  5. one all-to-all-v per buffer: run r goes to rank r, which stores the
     runs in source-rank order.  The received rows are exactly destination
     r's rows of the single-call layout (source rank, then token order);
     recv_src_idx holds each row's token index within its source rank.

combine sends every row back with the reverse all-to-all-v, into the send
buffer's layout, and reduces it with ep_combine on the send slots.

The library computes every layout, offset and row.  This module holds the
host logic between the steps and issues the collectives through
torch.distributed (NCCL between GPUs, gloo between CPU processes).  The
per-rank steps are a LocalSteps object: CudaSteps (the CUDA library, the
default) or any object with the same three methods, so that the exchange can
be run and checked on CPU ranks.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import (EPError, ShardLayout, alloc_dispatched, combine as ep_combine,
               dispatch as ep_dispatch, shard_layout, shard_offsets,
               shard_recv_tokens_per_expert)


class CudaSteps:
    """The per-rank steps on this process's GPU, through the CUDA library."""

    def layout(self, topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
               err: torch.Tensor | None = None) -> ShardLayout:
        return shard_layout(topk_idx, num_experts, num_ranks, err=err)

    def pack(self, x, topk_idx, topk_weights, layout: ShardLayout, rows: int, use_fp8: bool,
             err: torch.Tensor | None = None):
        """The send buffer: exactly `rows` rows (the layout's send_base[R])."""
        K = topk_idx.shape[1]
        out = alloc_dispatched(rows, x.shape[1], K, layout.num_experts, layout.num_ranks,
                               use_fp8, x.device)
        return ep_dispatch(x, topk_idx, topk_weights, layout, use_fp8=use_fp8, err=err, out=out)

    def combine(self, y_back, topk_idx, topk_weights, layout: ShardLayout,
                err: torch.Tensor | None = None):
        return ep_combine(y_back, topk_idx, topk_weights, layout, err=err)


class DistExchange:
    """The two collectives of the sharded form over a torch.distributed group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_gather_rows(self, row: torch.Tensor) -> torch.Tensor:
        """[n] on every rank -> [world, n], rank order."""
        out = [torch.empty_like(row) for _ in range(self.world)]
        self.dist.all_gather(out, row.contiguous(), group=self.group)
        return torch.stack(out)

    def all_to_all_rows(self, out: torch.Tensor, inp: torch.Tensor, out_splits, in_splits):
        """Rows of inp go out in runs of in_splits[r] to rank r; the runs from
        each rank land in out in rank order, out_splits[s] rows from rank s.
        Rows move as bytes, whatever their element type."""
        self.dist.all_to_all_single(_row_bytes(out), _row_bytes(inp), [int(v) for v in out_splits],
                                    [int(v) for v in in_splits], group=self.group)


def _row_bytes(t: torch.Tensor) -> torch.Tensor:
    """The same memory as [rows, bytes per row] uint8.  t must be contiguous
    (a received run must land in t itself, not in a copy); an empty t, which
    may carry any strides, becomes an empty byte tensor of the same width."""
    inner = 1
    for d in t.shape[1:]:
        inner *= int(d)
    if t.numel() == 0:
        return torch.empty((t.shape[0], inner * t.element_size()), dtype=torch.uint8,
                           device=t.device)
    if not t.is_contiguous():
        raise EPError("the exchange needs contiguous row buffers")
    return t.view(t.shape[0], inner).view(torch.uint8)


@dataclass
class ShardPlan:
    """Host-side offsets of one rank's exchange (shard_offsets)."""
    rank: int
    counts: np.ndarray         # [R, R] int32, counts[s][r] = tokens of rank s sent to rank r
    send_offsets: np.ndarray   # [R + 1] int64: this rank's run for rank r in its send buffer
    recv_offsets: np.ndarray   # [R + 1] int64: where rank s's run lands in the receive buffer

    @property
    def send_splits(self) -> np.ndarray:
        return np.diff(self.send_offsets)

    @property
    def recv_splits(self) -> np.ndarray:
        return np.diff(self.recv_offsets)

    @property
    def send_rows(self) -> int:
        return int(self.send_offsets[-1])

    @property
    def recv_rows(self) -> int:
        return int(self.recv_offsets[-1])


def make_plan(counts: np.ndarray, rank: int) -> ShardPlan:
    send, recv = shard_offsets(counts, rank)
    return ShardPlan(rank, np.ascontiguousarray(counts, np.int32), send, recv)


@dataclass
class ShardReceived:
    """What one rank receives: its rows of the single-call layout."""
    recv_x: torch.Tensor              # [rows, H] bf16, or uint8 E4M3 codes
    recv_scales: torch.Tensor | None  # [rows, H/128] float32 (FP8 only)
    recv_src_idx: torch.Tensor        # [rows] int32: token index within the source rank
    recv_topk_idx: torch.Tensor       # [rows, K] int64: local expert id, -1 elsewhere
    recv_topk_weights: torch.Tensor   # [rows, K] float32
    num_recv_tokens_per_expert: np.ndarray  # [E/R] int32 (host)
    recv_offsets: np.ndarray          # [R + 1]: rows from source rank s are [off[s], off[s+1])


@dataclass
class ShardHandle:
    """What combine needs from dispatch."""
    layout: ShardLayout
    plan: ShardPlan
    topk_idx: torch.Tensor
    topk_weights: torch.Tensor
    hidden: int


class ShardedEP:
    """dispatch / combine across the ranks of a process group, one rank per
    process.  `exchange` defaults to DistExchange over the default group and
    `steps` to CudaSteps."""

    def __init__(self, exchange=None, steps=None):
        self.ex = exchange if exchange is not None else DistExchange()
        self.steps = steps if steps is not None else CudaSteps()

    def dispatch(self, x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
                 num_experts: int, *, use_fp8: bool = False,
                 err: torch.Tensor | None = None) -> tuple[ShardReceived, ShardHandle]:
        R, rank = self.ex.world, self.ex.rank
        if num_experts % R:
            raise EPError("num_experts must be a multiple of the number of ranks")
        lay = self.steps.layout(topk_idx, num_experts, R, err=err)
        # the count exchange: a host-visible [R, R] matrix, as the notify step
        counts = self.ex.all_gather_rows(lay.send_counts).cpu().numpy()
        expert_counts = self.ex.all_gather_rows(lay.expert_counts).cpu().numpy()
        plan = make_plan(counts, rank)
        send = self.steps.pack(x, topk_idx, topk_weights, lay, plan.send_rows, use_fp8, err=err)
        H, K = x.shape[1], topk_idx.shape[1]
        n = plan.recv_rows
        dev = send.recv_x.device
        recv = ShardReceived(
            torch.empty((n, H), dtype=send.recv_x.dtype, device=dev),
            torch.empty((n, H // 128), dtype=torch.float32, device=dev) if use_fp8 else None,
            torch.empty(n, dtype=torch.int32, device=dev),
            torch.empty((n, K), dtype=torch.int64, device=dev),
            torch.empty((n, K), dtype=torch.float32, device=dev),
            shard_recv_tokens_per_expert(expert_counts, rank), plan.recv_offsets)
        pairs = [(recv.recv_x, send.recv_x), (recv.recv_src_idx, send.recv_src_idx),
                 (recv.recv_topk_idx, send.recv_topk_idx),
                 (recv.recv_topk_weights, send.recv_topk_weights)]
        if use_fp8:
            pairs.append((recv.recv_scales, send.recv_scales))
        for out, inp in pairs:
            self.ex.all_to_all_rows(out, inp[:plan.send_rows], plan.recv_splits, plan.send_splits)
        return recv, ShardHandle(lay, plan, topk_idx, topk_weights, H)

    def combine(self, y: torch.Tensor, handle: ShardHandle, *, weighted: bool = True,
                err: torch.Tensor | None = None) -> torch.Tensor:
        """y: [rows received, H] bf16 expert outputs in the receive buffer's
        row order.  Every row returns to its source rank, which reduces its
        tokens' rows (weighted by the top-k weights, or the rank sum)."""
        plan = handle.plan
        if y.shape[0] < plan.recv_rows:
            raise EPError(f"y must have the {plan.recv_rows} received rows, got {y.shape[0]}")
        # A rank that sent no rows (every one of its slots masked) still runs
        # the combine, which writes its zero rows and reads no row of y: one
        # placeholder row keeps y a real buffer.
        back = torch.empty((max(plan.send_rows, 1), y.shape[1]), dtype=y.dtype, device=y.device)
        self.ex.all_to_all_rows(back[:plan.send_rows], y[:plan.recv_rows], plan.send_splits,
                                plan.recv_splits)
        w = handle.topk_weights if weighted else None
        return self.steps.combine(back, handle.topk_idx, w, handle.layout, err=err)
