"""The five workloads at their full sizes, run exactly as bench.py runs them
(a captured CUDA graph of one decode step, replayed), with sampled
(request, KV head) units checked one by one against the oracle and
properties that hold at any size checked on every unit.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import (make_decoder, dev_bits, dev_status, host_bits, score_norm, assert_scores,
                      score_error_bound, assert_selection_valid, assert_attention, oracle_unit,
                      h2o_teacher_forced)

pytestmark = pytest.mark.gpu


def _graph_steps(dec, wl, steps, append, check):
    dec.q_buf.copy_(dev_bits(wl.q(0), wl.cfg.dtype))
    dec.capture(append=append)
    # capture does not execute; replay step by step
    for t in range(steps):
        dec.q_buf.copy_(dev_bits(wl.q(t), wl.cfg.dtype))
        if append:
            kn, vn = wl.kv_new(t)
            dec.k_buf.copy_(dev_bits(kn, wl.cfg.dtype))
            dec.v_buf.copy_(dev_bits(vn, wl.cfg.dtype))
        dec.replay()
        torch.cuda.synchronize()
        check(t)


def _check_page_units(dec, wl, t, steps_done, units, appended):
    """Teacher-forced checks of sampled (request, KV head) units after a step:
    page scores against the oracle's float64 scores of the same statistics;
    the oracle's top-k applied to the GPU's float32 scores equals the GPU's
    selection bit for bit; the selection is a valid top-k of the oracle's own
    scores within the float32 error bound; and the oracle's attention over
    the GPU's selection matches the GPU's output and lse on every unit."""
    c = wl.cfg
    qb = wl.q(t)
    scores = dec.scores.cpu().numpy()
    sel = dec.sel_idx.cpu().numpy()
    cnt = dec.sel_cnt.cpu().numpy()
    out = dec.out.float().cpu().numpy()
    lse = dec.lse.cpu().numpy()
    sc = c.scale if c.scale > 0 else O.default_scale(c.D)
    same = 0
    for b, h in units:
        r, ks, vs, qg, L = oracle_unit(wl, b, h, steps_done, qb[b])
        n = O.num_pages(L, c.ps)
        mn, mx, me = r["meta"]
        q = O.decode_kdt(qg, c.dtype)
        A = score_norm(mn, mx, me, q, c.w_avg, c.w_peak)
        # with a one-token append the step scores the tail beside the append:
        # that entry is unspecified (the tail is always selected)
        m = n - 1 if appended else n
        assert_scores(scores[b, h, :m], r["scores"][:m], A[:m])
        assert cnt[b, h] == min(c.topk, n)
        got_sel = sel[b, h, :cnt[b, h]]
        # A3 of the oracle on the GPU's own float32 scores (the tail's entry is never read)
        want_sel = O.select_pages(scores[b, h, :n].astype(np.float64), n, c.topk)
        assert np.array_equal(got_sel, want_sel), (b, h)
        assert_selection_valid(got_sel, r["scores"], score_error_bound(A, c.D, c.G), n, c.topk)
        same += int(np.array_equal(got_sel, r["sel"]))
        # A4 of the oracle over the GPU's selection
        pos = O.selected_positions(got_sel, L, c.ps)
        o, lw, _ = O.attention(q, O.decode_kdt(ks[pos], c.dtype), O.decode_kdt(vs[pos], c.dtype), sc)
        sl = slice(h * c.G, (h + 1) * c.G)
        assert_attention(out[b, sl], o, lse[b, sl], lw)
    return same


def _page_config(cid, steps, units_fn, append, check_steps=None):
    wl = make_workload(config(cid))
    dec = make_decoder(wl, stale="nan" if cid == 5 else "normal3")
    units = units_fn(wl)
    check_steps = set(check_steps if check_steps is not None else (0, steps - 1))

    def check(t):
        steps_done = t + 1 if append else 0
        if t in check_steps:
            _check_page_units(dec, wl, t, steps_done, units, append)
        cnt = dec.sel_cnt.cpu().numpy()
        sel = dec.sel_idx.cpu().numpy()
        out = dec.out.float()
        assert torch.isfinite(out).all()
        for b in range(wl.cfg.B):
            n = O.num_pages(wl.seq_len(b, steps_done), wl.cfg.ps)
            for h in range(wl.cfg.H_kv):
                s = sel[b, h, :cnt[b, h]]
                assert cnt[b, h] == min(wl.cfg.topk, n) and s[-1] == n - 1
                assert np.all(np.diff(s) > 0)

    _graph_steps(dec, wl, steps, append, check)
    assert dev_status(dec) == 0
    assert dec.seq_lens.cpu().tolist() == [wl.seq_len(b, steps if append else 0)
                                           for b in range(wl.cfg.B)]
    return dec, wl


def _all_units(wl):
    return [(b, h) for b in range(wl.cfg.B) for h in range(wl.cfg.H_kv)]


def test_full_tiny():
    _page_config(1, 1, _all_units, append=False)


def test_full_decode_loop():
    # every unit, every 8th step and the last
    _page_config(2, 64, _all_units, append=True, check_steps=list(range(0, 64, 8)) + [63])


def test_full_batched_gqa():
    units = [(0, 0), (2, 6), (5, 3), (7, 2), (9, 4), (11, 7), (13, 5), (15, 1)]
    _page_config(3, 2, lambda wl: units, append=False)


LONG_UNITS = [(0, 0), (0, 5), (1, 2), (1, 7), (2, 1), (2, 6), (3, 3), (3, 4)]


def test_full_long_context():
    dec, wl = _page_config(5, 32, lambda wl: LONG_UNITS, append=True)
    # meta of the pages the 32 appends touched, for a sampled unit
    b, h = 1, 4
    L = wl.seq_len(b, 32)
    ks = wl.k_seq(b, 32)[:, h, :]
    meta = host_bits(dec.cache.meta)
    for p in range(O.num_pages(wl.prefill_lens[b], 16) - 1, O.num_pages(L, 16)):
        rows = O.decode_kdt(ks[p * 16:min((p + 1) * 16, L)], "bf16")
        mn, mx, me = O.page_stats(rows, "bf16")
        blk = wl.block_table[b, p]
        got = [O.decode_kdt(meta[blk, h, i], "bf16") for i in range(3)]
        assert np.array_equal(got[0], mn) and np.array_equal(got[1], mx) and np.array_equal(got[2], me)


def test_full_token_h2o_teacher_forced():
    """The token-level workload at full size (8 requests x 8 KV heads, 4096-token
    prefill, all 256 decode steps, budget 512): eight units spread over
    requests and heads checked at every step against the oracle started from
    the GPU's pre-step state; bit-exact evictions on the GPU's own scores."""
    wl = make_workload(config(4))
    c = wl.cfg
    dec = make_decoder(wl)
    units = [(0, 0), (1, 3), (2, 6), (3, 1), (4, 4), (5, 7), (6, 2), (7, 5)]
    assert h2o_teacher_forced(dec, wl, units, c.decode_steps) == len(units) * c.decode_steps
    assert c.decode_steps == 256
    assert dev_status(dec) == 0


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_full_long_context_entmax(alpha):
    """The long-context workload with alpha-entmax over the selection, as
    bench.py --entmax runs it (graph replay, one-token appends): sampled units
    against the oracle's entmax attention over the GPU's own selection."""
    wl = make_workload(config(5))
    c = wl.cfg
    dec = make_decoder(wl, stale="nan", extra=dict(alpha=alpha))
    units = [(0, 0), (2, 5), (3, 7)]
    sc = c.scale if c.scale > 0 else O.default_scale(c.D)

    def check(t):
        out = dec.out.float()
        assert torch.isfinite(out).all() and torch.isfinite(dec.tau).all()
        if t not in (0, 3):
            return
        sel = dec.sel_idx.cpu().numpy()
        cnt = dec.sel_cnt.cpu().numpy()
        o_np = out.cpu().numpy()
        tau = dec.tau.cpu().numpy()
        lg = dec.logits.cpu().numpy()
        for b, h in units:
            L = wl.seq_len(b, t + 1)
            m = int(cnt[b, h])
            assert m == c.topk
            pos = O.selected_positions(sel[b, h, :m], L, c.ps)
            ks = O.decode_kdt(wl.k_seq(b, t + 1)[:, h, :][pos], c.dtype)
            vs = O.decode_kdt(wl.v_seq(b, t + 1)[:, h, :][pos], c.dtype)
            rows = slice(h * c.G, (h + 1) * c.G)
            q = O.decode_kdt(wl.q(t)[b, rows], c.dtype)
            o, _, z = O.attention_entmax(q, ks, vs, sc, alpha)
            assert_attention(o_np[b, rows], o)
            zg = lg[b, rows, :m * c.ps]
            zg = zg[:, np.isfinite(zg[0])].astype(np.float64)
            assert zg.shape == z.shape and np.all(np.abs(zg - z) <= 1e-4 * (1 + np.abs(z)))
            for gi in range(c.G):
                tz = O.entmax_threshold(zg[gi], alpha)
                assert abs(float(tau[b, h * c.G + gi]) - tz) <= 1e-6 * (1 + abs(tz))

    _graph_steps(dec, wl, 4, True, check)
    assert dev_status(dec) == 0


def test_full_long_context_gaussian():
    """The long-context workload with Gaussian-aware selection per query head
    (graph replay, one-token appends): sampled heads' moments, threshold and
    selection against the oracle, and the attention over the GPU's selection."""
    from test_gpu_gauss import _check_selection
    wl = make_workload(config(5))
    c = wl.cfg
    dec = make_decoder(wl, stale="nan", extra=dict(gaussian=True, alpha=1.5))
    heads = [(0, 0), (1, 17), (3, 63)]
    sc = c.scale if c.scale > 0 else O.default_scale(c.D)

    def check(t):
        assert torch.isfinite(dec.out.float()).all()
        cnt = dec.sel_cnt.cpu().numpy()
        assert np.all(cnt >= 1)
        if t not in (0, 2):
            return
        assert _check_selection(dec, wl, t + 1, wl.q(t), 1.5, heads) >= len(heads) - 1
        sel = dec.sel_idx.cpu().numpy()
        out = dec.out.float().cpu().numpy()
        for b, gq in heads:
            h = gq // c.G
            L = wl.seq_len(b, t + 1)
            pos = O.selected_positions(sel[b, gq, :cnt[b, gq]], L, c.ps)
            k = O.decode_kdt(wl.k_seq(b, t + 1)[:, h, :][pos], c.dtype)
            v = O.decode_kdt(wl.v_seq(b, t + 1)[:, h, :][pos], c.dtype)
            o, _, _ = O.attention_entmax(O.decode_kdt(wl.q(t)[b, gq], c.dtype)[None], k, v, sc, 1.5)
            assert_attention(out[b, gq][None], o)

    _graph_steps(dec, wl, 3, True, check)
    assert dev_status(dec) == 0
