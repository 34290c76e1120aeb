"""Per-query-head selection ([entmax] "Top-k": pages kept per query head) on
the GPU against the oracle: each query head's scores (the oracle's page score
with a group of one), a valid top-k per query head, and each head's attention
over exactly its own selected pages.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import (make_decoder, dev_bits, dev_status, step_inputs, score_norm, assert_scores,
                      score_error_bound, assert_selection_valid, assert_attention)

pytestmark = pytest.mark.gpu


def _head_oracle(wl, b, g, steps_done, q_bits):
    """Scores, score scale and length for query head g of request b."""
    c = wl.cfg
    h = g // c.G
    L = wl.seq_len(b, steps_done)
    mn, mx, me = O.head_meta(wl.k_seq(b, steps_done)[:, h, :], L, c.ps, c.dtype)
    q = O.decode_kdt(q_bits[g:g + 1], c.dtype)
    return O.score_pages(mn, mx, me, q, c.w_avg, c.w_peak), score_norm(mn, mx, me, q, c.w_avg, c.w_peak), L


@pytest.mark.parametrize("cid,G,D", [(1, 4, 64), (2, 4, 128), (3, 4, 128), (3, 1, 128), (3, 16, 64),
                                      (5, 8, 128)])
def test_per_head_scores_selection_and_attention(cid, G, D):
    cfg = config(cid, small=True)
    cfg = cfg.replace(H_q=cfg.H_kv * G, D=D)
    wl = make_workload(cfg)
    c = wl.cfg
    dec = make_decoder(wl, extra=dict(per_query_head=True))
    steps = min(wl.total_steps, 3)
    for t in range(max(steps, 1)):
        if steps:
            q, kn, vn = step_inputs(wl, t)
            dec.step(q, kn, vn)
            done = t + 1
        else:
            q = dev_bits(wl.q(0), c.dtype)
            dec.step(q)
            done = 0
        torch.cuda.synchronize()
        qb = wl.q(t)
        scores = dec.scores.cpu().numpy()
        sel, cnt = dec.sel_idx.cpu().numpy(), dec.sel_cnt.cpu().numpy()
        out, lse = dec.out.float().cpu().numpy(), dec.lse.cpu().numpy()
        for b in range(c.B):
            for g in range(c.H_q):
                S, A, L = _head_oracle(wl, b, g, done, qb[b])
                n = O.num_pages(L, c.ps)
                assert_scores(scores[b, g, :n], S, A)
                got = sel[b, g, :cnt[b, g]]
                assert cnt[b, g] == min(c.topk, n)
                assert_selection_valid(got, S, score_error_bound(A, c.D, 1), n, c.topk)
                # this head's attention over exactly the pages it selected
                h = g // c.G
                pos = O.selected_positions(got, L, c.ps)
                ks = O.decode_kdt(wl.k_seq(b, done)[pos, h, :], c.dtype)
                vs = O.decode_kdt(wl.v_seq(b, done)[pos, h, :], c.dtype)
                qq = O.decode_kdt(qb[b, g:g + 1], c.dtype)
                o, l, _ = O.attention(qq, ks, vs, c.scale if c.scale > 0 else O.default_scale(c.D))
                assert_attention(out[b, g:g + 1], o, lse[b, g:g + 1], l)
    assert dev_status(dec) == 0


def test_per_head_agrees_with_group_of_one():
    """With G = 1 per-query-head and per-KV-head selection compute the same
    thing (the scorers by different arithmetic: tensor-core products for the
    per-head rows): scores within float32 rounding of each other, and where the
    selections agree the attention outputs are bit-identical."""
    cfg = config(3, small=True).replace(H_q=2, H_kv=2)
    wl = make_workload(cfg)
    a = make_decoder(wl, extra=dict(per_query_head=True))
    b = make_decoder(wl)
    q = dev_bits(wl.q(0), cfg.dtype)
    a.attend(q)
    b.attend(q)
    torch.cuda.synchronize()
    for r in range(cfg.B):                      # entries past a request's pages are untouched
        n = O.num_pages(int(wl.prefill_lens[r]), cfg.ps)
        sa, sb = a.scores[r, :, :n].cpu().numpy(), b.scores[r, :, :n].cpu().numpy()
        assert np.all(np.abs(sa - sb) <= 1e-5 * np.maximum(np.abs(sb), 1.0))
    same = 0
    for r in range(cfg.B):
        for h in range(cfg.H_kv):
            if torch.equal(a.sel_idx[r, h], b.sel_idx[r, h]):
                same += 1
                assert torch.equal(a.out[r, h].view(torch.int16), b.out[r, h].view(torch.int16))
                assert torch.equal(a.lse[r, h].view(torch.int32), b.lse[r, h].view(torch.int32))
    assert same >= cfg.B * cfg.H_kv // 2


@pytest.mark.parametrize("G", [8, 16])
def test_per_head_scores_bad_block_and_overflow(G):
    """A page with an out-of-range block id scores NaN for every head of its
    KV head and sets SA_DEV_BAD_BLOCK; a request longer than its block-table
    row sets SA_DEV_OVERFLOW and is scored up to the row's end; every other
    page's scores match the oracle."""
    from sparse_paged_kv_page_gb300 import sa_score_pages_qh
    from sparse_paged_kv_page_gb300._lib import SA_DEV_BAD_BLOCK, SA_DEV_OVERFLOW
    cfg = config(3, small=True)
    cfg = cfg.replace(H_q=cfg.H_kv * G)
    wl = make_workload(cfg)
    c = wl.cfg
    dec = make_decoder(wl, extra=dict(per_query_head=True))
    q = dev_bits(wl.q(0), c.dtype)
    lens, bt = dec.seq_lens.clone(), dec.block_table.clone()
    dec.block_table[1, 1] = wl.num_blocks + 3
    dec.seq_lens[0] = dec.block_table.shape[1] * c.ps + 50
    dec.scores.fill_(7.0)
    sa_score_pages_qh(dec.cache.struct, dec.batch, q, c.H_q, c.w_avg, c.w_peak, dec.scores, dec.max_pages,
                      dev_status=dec.dev_status)
    torch.cuda.synchronize()
    st = dev_status(dec)
    assert st & SA_DEV_BAD_BLOCK and st & SA_DEV_OVERFLOW
    scores = dec.scores.cpu().numpy()
    row = dec.block_table.shape[1]
    assert np.all(scores[0, :, :row] != 7.0)                # the overflowing request: its whole row scored
    for b in (1, 2):
        for g in range(c.H_q):
            S, A, L = _head_oracle(wl, b, g, 0, wl.q(0)[b])
            n = O.num_pages(L, c.ps)
            got = scores[b, g, :n]
            if b == 1:
                assert np.isnan(got[1])
                keep = np.arange(n) != 1
                assert_scores(got[keep], S[keep], A[keep])
            else:
                assert_scores(got, S, A)
    dec.block_table.copy_(bt)
    dec.seq_lens.copy_(lens)
