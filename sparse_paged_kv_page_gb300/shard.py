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
single GPU; `gather_slices` is the exchange when the shards live on
different ranks (torch.distributed all-gather, plumbing only).
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
    """All-gather of equally shaped per-rank slices, concatenated along `dim`
    in rank order (the score rows of a sharded step)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(parts, local.contiguous(), group=group)
    return torch.cat(parts, dim=dim)


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
