"""Sequence sharding of the read path of a page-level decode step.

Every request's pages are split into contiguous ranges, one per shard. Each
shard scores its own pages, the score slices are gathered into whole rows
(the one exchange of the step: an all-gather across devices, a copy into one
row here), one top-k runs over the whole rows (tail forced), and each shard
attends its part of the selection; the partial states are merged by
log-sum-exp. With identical page scores the selection equals the unsharded
one bit for bit, and the merge is exact up to rounding ("MergeAttnStates" of
the vllm.cpp chunked-context test; "EntmaxKV" README, Top-k).

`SequenceShards` runs all shards of one cache on one device (each shard a
view of its page range), which is how the sharded path is exercised on a
single GPU. When the shards live on different ranks the step has two
exchanges (torch.distributed all-gathers, plumbing only): `gather_slices`
joins the score slices of every rank's page range (ranges may differ by a
page) into whole rows before the selection, and `gather_states` collects every
rank's partial (o, lse) for `sa_merge_states` (`merge_across_ranks`).

KV-head partitioning needs no exchange at all: a rank holding KV heads
[h0, h1) keeps those heads' pool and statistics slices and their G query
heads each, and decodes them exactly as the whole cache would
(`kv_head_slice`, `query_head_slice`); the rows of the heads it holds are the
output of the step for those heads.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import torch

from .api import (alloc_decode_workspace, batch_view, sa_merge_states, sa_score_pages,
                  sa_select_topk, sa_shard_lengths, sa_shard_selection, sa_sparse_decode)


def page_ranges(num_pages: int, num_shards: int) -> List[Tuple[int, int]]:
    """Contiguous page ranges [lo, hi) covering [0, num_pages), as equal as possible."""
    if num_shards <= 0 or num_pages <= 0:
        raise ValueError("need at least one page and one shard")
    base, extra = divmod(num_pages, num_shards)
    out, lo = [], 0
    for s in range(num_shards):
        hi = lo + base + (1 if s < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def gather_slices(local: torch.Tensor, dim: int, group=None) -> torch.Tensor:
    """All-gather of per-rank slices along `dim`, concatenated in rank order
    (the score rows of a sequence-sharded step: each rank's page range, whose
    widths may differ, e.g. 2732 / 2731 / 2731). The widths are exchanged
    first; every slice is padded to the widest for the gather and trimmed after."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    width = torch.tensor([local.shape[dim]], dtype=torch.int64, device=local.device)
    widths = [torch.zeros_like(width) for _ in range(world)]
    dist.all_gather(widths, width, group=group)
    widths = [int(w.item()) for w in widths]
    shape = list(local.shape)
    shape[dim] = max(widths)
    buf = local.new_zeros(shape)
    buf.narrow(dim, 0, local.shape[dim]).copy_(local)
    parts = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(parts, buf, group=group)
    return torch.cat([p.narrow(dim, 0, w) for p, w in zip(parts, widths)], dim=dim)


def gather_states(o_part: torch.Tensor, lse_part: torch.Tensor, group=None):
    """All-gather every rank's partial attention state -- o [..., D] and lse
    [...] over its own page range (lse = -inf where it attended nothing) --
    stacked in rank order: ([world, ...D], [world, ...]), the o_parts /
    lse_parts layout of sa_merge_states."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    o_all = [torch.empty_like(o_part) for _ in range(world)]
    l_all = [torch.empty_like(lse_part) for _ in range(world)]
    dist.all_gather(o_all, o_part.contiguous(), group=group)
    dist.all_gather(l_all, lse_part.contiguous(), group=group)
    return torch.stack(o_all), torch.stack(l_all)


def merge_across_ranks(o_part: torch.Tensor, lse_part: torch.Tensor, out: torch.Tensor,
                       lse: torch.Tensor = None, group=None):
    """The second exchange of a sequence-sharded step on several ranks: gather
    the partial states, then merge them by log-sum-exp on this rank's device
    (sa_merge_states). o_part [B, H_q, D] (bf16/fp16), lse_part [B, H_q] float32."""
    o_parts, lse_parts = gather_states(o_part, lse_part, group)
    rows = o_part.numel() // o_part.shape[-1]
    sa_merge_states(o_parts, lse_parts, o_parts.shape[0], rows, o_part.shape[-1], out, lse=lse)
    return out


def kv_head_range(num_kv_heads: int, num_ranks: int, rank: int) -> Tuple[int, int]:
    """KV heads [h0, h1) held by `rank` when the heads are partitioned (as equal as possible)."""
    return page_ranges(num_kv_heads, num_ranks)[rank]


def kv_head_slice(t: torch.Tensor, h0: int, h1: int, head_axis: int = 1) -> torch.Tensor:
    """The rows of KV heads [h0, h1) of a pool ([num_blocks, H_kv, ps, D]),
    statistics ([num_blocks, H_kv, 3, D]) or per-token score ([slots, H_kv],
    head_axis = 1 as well) tensor, as the contiguous tensor a rank holding
    those heads keeps."""
    return t.narrow(head_axis, h0, h1 - h0).contiguous()


def query_head_slice(q: torch.Tensor, h0: int, h1: int, group_size: int) -> torch.Tensor:
    """The query heads of KV heads [h0, h1) (each KV head's G consecutive
    query heads) of q [B, H_q, D]."""
    return q.narrow(1, h0 * group_size, (h1 - h0) * group_size).contiguous()


class SequenceShards:
    """The read path (score -> select -> attend) of a page-level decoder with
    its pages split over `num_shards` page ranges of the same cache."""

    def __init__(self, dec, num_shards: int):
        if dec.token_level or dec.qh or getattr(dec, "entmax", False) or getattr(dec, "gaussian", False):
            raise ValueError("sequence sharding is built for the page-level softmax step")
        self.dec = dec
        self.S = num_shards
        self.ranges = page_ranges(dec.max_pages, num_shards)
        B, H, Hq, D = dec.B, dec.H_kv, dec.H_q, dec.D
        i32 = dict(dtype=torch.int32, device=dec.device)
        self.lens = [torch.zeros((B,), **i32) for _ in range(num_shards)]
        self.batches = [batch_view(dec.block_table, self.lens[s], lo) for s, (lo, _) in enumerate(self.ranges)]
        self.local_scores = [torch.empty((B, H, hi - lo), dtype=torch.float32, device=dec.device)
                             for lo, hi in self.ranges]
        self.scores = torch.empty((B, H, dec.max_pages), dtype=torch.float32, device=dec.device)
        self.sel_idx = torch.zeros((B, H, dec.topk), **i32)
        self.sel_cnt = torch.zeros((B, H), **i32)
        self.shard_idx = [torch.zeros((B, H, dec.topk), **i32) for _ in range(num_shards)]
        self.shard_cnt = [torch.zeros((B, H), **i32) for _ in range(num_shards)]
        self.o_parts = torch.empty((num_shards, B, Hq, D), dtype=dec.dtype, device=dec.device)
        self.lse_parts = torch.empty((num_shards, B, Hq), dtype=torch.float32, device=dec.device)
        self.workspaces = [alloc_decode_workspace(B, H, Hq, D, dec.ps, dec.topk, dec.device)
                           for _ in range(num_shards)]
        self.out = torch.empty((B, Hq, D), dtype=dec.dtype, device=dec.device)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=dec.device)

    def attend(self, q: torch.Tensor):
        d = self.dec
        B, H = d.B, d.H_kv
        for s, (lo, hi) in enumerate(self.ranges):
            sa_shard_lengths(d.seq_lens, B, d.ps, lo, hi, self.lens[s])
            sa_score_pages(d.cache.struct, self.batches[s], q, d.H_q, d.w_avg, d.w_peak,
                           self.local_scores[s], hi - lo, dev_status=d.dev_status)
        # the exchange: every shard's slice into the whole rows
        for s, (lo, hi) in enumerate(self.ranges):
            self.scores[:, :, lo:hi].copy_(self.local_scores[s])
        sa_select_topk(self.scores, d.max_pages, d.batch, d.ps, H, d.topk, self.sel_idx, self.sel_cnt,
                       dev_status=d.dev_status)
        for s, (lo, hi) in enumerate(self.ranges):
            sa_shard_selection(self.sel_idx, self.sel_cnt, d.topk, B * H, lo, hi, self.shard_idx[s],
                               self.shard_cnt[s], d.topk, dev_status=d.dev_status)
            sa_sparse_decode(d.cache.struct, self.batches[s], q, d.H_q, self.shard_idx[s],
                             self.shard_cnt[s], d.topk, d.scale, self.o_parts[s], lse=self.lse_parts[s],
                             workspace=self.workspaces[s], dev_status=d.dev_status)
        sa_merge_states(self.o_parts, self.lse_parts, self.S, B * d.H_q, d.D, self.out, lse=self.lse)
        return self.out
