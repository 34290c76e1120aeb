"""Sequence sharding of the page-level read path on one GPU: every request's
pages split over S page ranges of one cache, each range scored and attended
as its own shard, one top-k over the gathered score rows, the partial states
merged by log-sum-exp ("MergeAttnStates" of the vllm.cpp chunked-context
test). The scores and the selection must equal the unsharded step's bit for
bit; the output must match the oracle's attention over that selection.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import make_decoder, dev_bits, dev_status, host_bits, assert_attention

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cid,S", [(5, 2), (5, 3), (3, 4), (2, 5), (1, 3)])
def test_sharded_step_equals_the_unsharded_one(cid, S):
    from sparse_paged_kv_page_gb300.shard import SequenceShards
    wl = make_workload(config(cid, small=True))
    c = wl.cfg
    dec = make_decoder(wl)
    sh = SequenceShards(dec, S)
    q = dev_bits(wl.q(0), c.dtype)
    out_s = sh.attend(q).clone()
    lse_s = sh.lse.clone()
    dec.attend(q)
    torch.cuda.synchronize()
    scores_d, scores_s = dec.scores.cpu().numpy(), sh.scores.cpu().numpy()
    for b in range(c.B):
        n = O.num_pages(int(wl.prefill_lens[b]), c.ps)
        assert np.array_equal(scores_d[b, :, :n].view(np.uint32), scores_s[b, :, :n].view(np.uint32))
    assert torch.equal(dec.sel_cnt, sh.sel_cnt)
    for b in range(c.B):
        for h in range(c.H_kv):
            k = int(dec.sel_cnt[b, h])
            assert torch.equal(dec.sel_idx[b, h, :k], sh.sel_idx[b, h, :k])
    # every selected page went to exactly one shard
    got = sum(int(x.sum()) for x in sh.shard_cnt)
    assert got == int(sh.sel_cnt.sum())
    # the merged output against the oracle over the same selection
    sel = sh.sel_idx.cpu().numpy()
    cnt = sh.sel_cnt.cpu().numpy()
    o = out_s.float().cpu().numpy()
    lse = lse_s.cpu().numpy()
    sc = c.scale if c.scale > 0 else O.default_scale(c.D)
    qb = wl.q(0)
    for b in range(c.B):
        L = int(wl.prefill_lens[b])
        for h in range(c.H_kv):
            pos = O.selected_positions(sel[b, h, :cnt[b, h]], L, c.ps)
            k = O.decode_kdt(wl.k_seq(b)[:, h, :][pos], c.dtype)
            v = O.decode_kdt(wl.v_seq(b)[:, h, :][pos], c.dtype)
            rows = slice(h * c.G, (h + 1) * c.G)
            ow, lw, _ = O.attention(O.decode_kdt(qb[b, rows], c.dtype), k, v, sc)
            assert_attention(o[b, rows], ow, lse[b, rows], lw)
    assert dev_status(dec) == 0


def test_merge_states_against_the_oracle():
    from sparse_paged_kv_page_gb300 import sa_merge_states
    rng = np.random.default_rng(3)
    S, rows, D = 4, 37, 128
    o_parts = rng.standard_normal((S, rows, D)).astype(np.float32)
    lse = rng.normal(0, 3, size=(S, rows)).astype(np.float32)
    lse[1, :5] = -np.inf                                   # empty parts
    lse[:, 7] = -np.inf                                    # every part empty
    lse[2, 9] = np.inf                                     # counted as empty
    ob = torch.from_numpy(o_parts).to(torch.bfloat16).cuda()
    out = torch.empty((rows, D), dtype=torch.bfloat16, device="cuda")
    lse_out = torch.empty(rows, device="cuda")
    sa_merge_states(ob, torch.from_numpy(lse).cuda(), S, rows, D, out, lse=lse_out)
    torch.cuda.synchronize()
    o_in = ob.float().cpu().numpy().astype(np.float64)
    want = np.zeros((rows, D)); wl = np.zeros(rows)
    for r in range(rows):
        w_o, w_l = O.merge_partials(o_in[:, r][:, None, :], lse[:, r][:, None])
        want[r], wl[r] = w_o[0], w_l[0]
    assert_attention(out.float().cpu().numpy(), want, lse_out.cpu().numpy(), wl, atol=1e-2, rtol=1e-2)
    # every part empty: part 0's output passes through ("MergeAttnStates", the prefix output)
    assert torch.equal(out[7], ob[0, 7]) and lse_out[7].item() == -np.inf


def test_shard_selection_splits_in_order():
    from sparse_paged_kv_page_gb300 import sa_shard_selection
    sel = torch.tensor([[0, 3, 4, 9, 10, 15, -1, -1], [2, 5, 6, 7, 8, 11, 12, 13]], dtype=torch.int32,
                       device="cuda")
    cnt = torch.tensor([6, 8], dtype=torch.int32, device="cuda")
    ranges = [(0, 5), (5, 10), (10, 16)]
    want = [[[0, 3, 4], [2]], [[4], [0, 1, 2, 3]], [[0, 5], [1, 2, 3]]]
    for (lo, hi), w in zip(ranges, want):
        idx = torch.full((2, 8), -7, dtype=torch.int32, device="cuda")
        c = torch.zeros(2, dtype=torch.int32, device="cuda")
        sa_shard_selection(sel, cnt, 8, 2, lo, hi, idx, c, 8)
        torch.cuda.synchronize()
        for u in range(2):
            assert idx[u, :int(c[u])].tolist() == w[u]


def test_sharded_step_with_an_empty_request_and_empty_shards():
    """Ragged requests over many shards leave some shards with no pages of a
    request (and one request with none at all): those parts carry lse = -inf
    and the merge still matches the unsharded step."""
    from sparse_paged_kv_page_gb300.shard import SequenceShards
    wl = make_workload(config(3, small=True))
    c = wl.cfg
    dec = make_decoder(wl)
    dec.seq_lens[1] = 0
    sh = SequenceShards(dec, 7)
    q = dev_bits(wl.q(0), c.dtype)
    out_s = sh.attend(q).clone()
    lse_s = sh.lse.clone()
    dec.attend(q)
    torch.cuda.synchronize()
    assert torch.equal(dec.sel_cnt, sh.sel_cnt) and int(sh.sel_cnt[1].abs().sum()) == 0
    assert torch.all(out_s[1].float() == 0) and torch.all(lse_s[1] == -float("inf"))
    for b in (0, 2):
        ok = torch.isfinite(dec.lse[b])
        assert torch.allclose(lse_s[b][ok], dec.lse[b][ok], atol=1e-3)
        assert torch.allclose(out_s[b].float(), dec.out[b].float(), atol=2e-2, rtol=2e-2)
    assert dev_status(dec) == 0


def test_kv_head_partition_reproduces_the_whole_step():
    """KV-head partitioning has no exchange: a decoder holding only KV heads
    [h0, h1) -- their pool and statistics slices, their G query heads each --
    reproduces the whole decoder's scores, selection, output and lse rows for
    those heads bit for bit (the same per-(page, head) arithmetic, and here the
    same split count per unit)."""
    from sparse_paged_kv_page_gb300.shard import kv_head_range, kv_head_slice, query_head_slice
    from sparse_paged_kv_page_gb300.step import SparseDecoder
    wl = make_workload(config(5, small=True))
    c = wl.cfg
    dec = make_decoder(wl)
    q = dev_bits(wl.q(0), c.dtype)
    dec.step(q)
    torch.cuda.synchronize()
    lens = dec.seq_lens.cpu().numpy()
    for r in range(2):
        h0, h1 = kv_head_range(c.H_kv, 2, r)
        part = SparseDecoder(batch=c.B, num_q_heads=(h1 - h0) * c.G, num_kv_heads=h1 - h0,
                             head_dim=c.D, page_size=c.ps, num_blocks=wl.num_blocks,
                             bt_stride=wl.max_pages, dtype=dec.dtype, scale=c.scale, topk=c.topk,
                             w_avg=c.w_avg, w_peak=c.w_peak)
        part.cache.k.copy_(kv_head_slice(dec.cache.k, h0, h1))
        part.cache.v.copy_(kv_head_slice(dec.cache.v, h0, h1))
        part.cache.meta.copy_(kv_head_slice(dec.cache.meta, h0, h1))
        part.set_block_table(torch.from_numpy(wl.block_table))
        part.seq_lens.copy_(dec.seq_lens)
        part.step(query_head_slice(q, h0, h1, c.G))
        torch.cuda.synchronize()
        rows = slice(h0 * c.G, h1 * c.G)
        for b in range(c.B):
            n = O.num_pages(int(lens[b]), c.ps)
            assert torch.equal(part.scores[b, :, :n].view(torch.int32),
                               dec.scores[b, h0:h1, :n].view(torch.int32))
        assert torch.equal(part.sel_cnt, dec.sel_cnt[:, h0:h1])
        for b in range(c.B):
            for hh in range(h1 - h0):
                k = int(part.sel_cnt[b, hh])
                assert torch.equal(part.sel_idx[b, hh, :k], dec.sel_idx[b, h0 + hh, :k])
        assert torch.equal(part.out.view(torch.int16), dec.out[:, rows].view(torch.int16))
        assert torch.equal(part.lse.view(torch.int32), dec.lse[:, rows].view(torch.int32))
        assert dev_status(part) == 0
    assert dev_status(dec) == 0
