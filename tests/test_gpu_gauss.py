"""Gaussian-aware selection ("EntmaxKV" README, How it works) on the GPU
against the oracle.

* k_std written by the append (prefill and decode steps) equals the oracle's
  once-rounded population std of the page's valid keys;
* the page moments m_p, v_p of every query head agree with the oracle's within
  float32 rounding, tau_hat within 1e-4, and the selection is the oracle's
  except for pages whose margin to tau_hat is within the float32 error of the
  estimate; the tail page is always kept, indices ascend, counts match;
* sa_sparse_decode_entmax_qh on random per-head selections, and the whole
  Gaussian-aware step on the GPU's own selection, match the oracle's entmax
  attention.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import make_decoder, dev_bits, dev_status, host_bits, assert_attention, step_inputs

pytestmark = pytest.mark.gpu


def _scale(c):
    return c.scale if c.scale > 0 else O.default_scale(c.D)


def _gauss_decoder(cid, alpha=1.5, small=True, stale="normal3", **kw):
    wl = make_workload(config(cid, small=small).replace(**kw) if kw else config(cid, small=small))
    dec = make_decoder(wl, stale=stale, extra=dict(gaussian=True, alpha=alpha))
    return wl, dec


def _check_kstd(dec, wl, steps_done):
    c = wl.cfg
    got = host_bits(dec.cache.kstd)
    for b in range(c.B):
        L = wl.seq_len(b, steps_done)
        ks = wl.k_seq(b, steps_done)
        for h in range(c.H_kv):
            _, sd, _ = O.head_gauss_stats(ks[:, h, :], L, c.ps, c.dtype)
            blk = wl.block_table[b, :O.num_pages(L, c.ps)]
            g = O.decode_kdt(got[blk, h], c.dtype)
            assert np.array_equal(g, sd), (b, h, np.argwhere(g != sd)[:4])


@pytest.mark.parametrize("cid", [2, 3, 5])
def test_kstd_after_prefill_and_appends(cid):
    wl, dec = _gauss_decoder(cid)
    _check_kstd(dec, wl, 0)
    for t in range(min(wl.total_steps, 20)):
        dec.append(*step_inputs(wl, t)[1:])
    torch.cuda.synchronize()
    _check_kstd(dec, wl, min(wl.total_steps, 20))
    assert dev_status(dec) == 0


def _oracle_head(wl, b, gq, steps_done, q_bits, alpha):
    c = wl.cfg
    h = gq // c.G
    L = wl.seq_len(b, steps_done)
    return O.gauss_decode_unit(wl.k_seq(b, steps_done)[:, h, :], wl.v_seq(b, steps_done)[:, h, :], L,
                               q_bits[b, gq], ps=c.ps, alpha=alpha, dtype=c.dtype, scale=c.scale)


def _check_selection(dec, wl, steps_done, q_bits, alpha, heads):
    """Moments, tau_hat and the selection of the given (request, query head)s."""
    c = wl.cfg
    mom = dec.moments.cpu().numpy()
    th = dec.tau_hat.cpu().numpy()
    sel = dec.sel_idx.cpu().numpy()
    cnt = dec.sel_cnt.cpu().numpy()
    same = 0
    for b, gq in heads:
        r = _oracle_head(wl, b, gq, steps_done, q_bits, alpha)
        n = len(r["m"])
        m, v = mom[b, gq, :n, 0].astype(np.float64), mom[b, gq, :n, 1].astype(np.float64)
        qd = np.abs(O.decode_kdt(q_bits[b, gq], c.dtype))
        tol_m = 1e-5 * _scale(c) * (np.abs(r["mean"]) @ qd) + 1e-9   # float32 error of the dot product
        assert np.all(np.abs(m - r["m"]) <= tol_m), (b, gq)
        assert np.all(np.abs(v - r["v"]) <= 1e-5 * r["v"] + 1e-9), (b, gq)
        assert abs(float(th[b, gq]) - r["tau_hat"]) <= 1e-4 * (1 + abs(r["tau_hat"])), (b, gq)
        got = sel[b, gq, :cnt[b, gq]]
        assert got[-1] == n - 1 and np.all(np.diff(got) > 0)
        # pages away from the threshold must agree with the oracle
        kappa = np.array([O.gauss_max_factor(int(f)) for f in r["fill"]])
        margin = (alpha - 1) * (r["m"] + kappa * np.sqrt(r["v"])) - r["tau_hat"]
        tol = 1e-4 * (1 + abs(r["tau_hat"])) + (alpha - 1) * (tol_m + kappa * 1e-5 * np.sqrt(r["v"]))
        firm = np.abs(margin) > tol
        firm[n - 1] = True
        want = np.zeros(n, bool); want[r["sel"]] = True
        have = np.zeros(n, bool); have[got] = True
        assert np.array_equal(want[firm], have[firm]), (b, gq)
        same += int(np.array_equal(want, have))
    return same


@pytest.mark.parametrize("cid,alpha", [(5, 1.5), (5, 2.0), (3, 1.5), (2, 2.0)])
def test_gaussian_step_against_the_oracle(cid, alpha):
    wl, dec = _gauss_decoder(cid, alpha)
    c = wl.cfg
    heads = [(b, gq) for b in range(c.B) for gq in range(c.H_q)]
    steps = min(wl.total_steps, 3)
    sc = _scale(c)
    for t in range(steps):
        q, kn, vn = step_inputs(wl, t)
        dec.step(q, kn, vn)
        torch.cuda.synchronize()
        qb = wl.q(t)
        same = _check_selection(dec, wl, t + 1, qb, alpha, heads)
        assert same >= 0.9 * len(heads), (same, len(heads))
        # attention over the GPU's own selection
        sel = dec.sel_idx.cpu().numpy()
        cnt = dec.sel_cnt.cpu().numpy()
        out = dec.out.float().cpu().numpy()
        tau = dec.tau.cpu().numpy()
        for b, gq in heads:
            h = gq // c.G
            L = wl.seq_len(b, t + 1)
            pos = O.selected_positions(sel[b, gq, :cnt[b, gq]], L, c.ps)
            k = O.decode_kdt(wl.k_seq(b, t + 1)[:, h, :][pos], c.dtype)
            v = O.decode_kdt(wl.v_seq(b, t + 1)[:, h, :][pos], c.dtype)
            qq = O.decode_kdt(qb[b, gq], c.dtype)[None]
            o, tz, _ = O.attention_entmax(qq, k, v, sc, alpha)
            assert_attention(out[b, gq][None], o)
            assert abs(float(tau[b, gq]) - tz[0]) <= 1e-4 * (1 + abs(tz[0]))
    assert dev_status(dec) == 0


def test_entmax_qh_on_random_per_head_selections():
    from sparse_paged_kv_page_gb300 import sa_sparse_decode_entmax_qh, alloc_entmax_workspace
    wl = make_workload(config(5, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    rng = np.random.default_rng(17)
    k = 20
    sel = np.zeros((c.B, c.H_q, k), np.int64)
    cnt = np.zeros((c.B, c.H_q), np.int64)
    for b in range(c.B):
        n = O.num_pages(int(wl.prefill_lens[b]), c.ps)
        for g in range(c.H_q):
            m = int(rng.integers(1, k + 1))
            pick = np.sort(np.append(rng.choice(n - 1, size=m - 1, replace=False), n - 1))
            sel[b, g, :m] = pick
            cnt[b, g] = m
    out = torch.empty((c.B, c.H_q, c.D), dtype=dec.dtype, device="cuda")
    tau = torch.empty((c.B, c.H_q), device="cuda")
    ws = alloc_entmax_workspace(c.B, c.H_q, c.H_q, c.D, c.ps, k)
    qb = wl.q(0)
    sa_sparse_decode_entmax_qh(dec.cache.struct, dec.batch, dev_bits(qb, c.dtype), c.H_q,
                               torch.from_numpy(sel.astype(np.int32)).cuda(),
                               torch.from_numpy(cnt.astype(np.int32)).cuda(), k, 1.5, dec.scale, out,
                               tau=tau, workspace=ws, dev_status=dec.dev_status)
    torch.cuda.synchronize()
    o_np = out.float().cpu().numpy()
    sc = _scale(c)
    for b in range(c.B):
        L = int(wl.prefill_lens[b])
        for g in range(c.H_q):
            h = g // c.G
            pos = O.selected_positions(sel[b, g, :cnt[b, g]], L, c.ps)
            kk = O.decode_kdt(wl.k_seq(b)[:, h, :][pos], c.dtype)
            vv = O.decode_kdt(wl.v_seq(b)[:, h, :][pos], c.dtype)
            o, tz, _ = O.attention_entmax(O.decode_kdt(qb[b, g], c.dtype)[None], kk, vv, sc, 1.5)
            assert_attention(o_np[b, g][None], o)
    assert dev_status(dec) == 0


def test_gauss_select_rejects_before_launching():
    from sparse_paged_kv_page_gb300 import SaError, sa_gauss_select
    wl, dec = _gauss_decoder(5)
    c = wl.cfg
    q = dev_bits(wl.q(0), c.dtype)
    args = (dec.cache.struct, dec.batch, q, c.H_q)
    with pytest.raises(SaError) as e:                          # no closed form for this alpha
        sa_gauss_select(*args, 1.25, dec.scale, dec.moments, dec.max_pages, dec.sel_idx,
                        dec.sel_cnt, dec.sel_stride)
    assert e.value.status == 2
    with pytest.raises(SaError) as e:                          # a selection too short for every page
        sa_gauss_select(*args, 1.5, dec.scale, dec.moments, dec.max_pages, dec.sel_idx,
                        dec.sel_cnt, dec.max_pages - 1)
    assert e.value.status == 1
    plain = make_decoder(wl)                                   # a cache without k_std
    with pytest.raises(SaError) as e:
        sa_gauss_select(plain.cache.struct, plain.batch, q, c.H_q, 1.5, dec.scale, dec.moments,
                        dec.max_pages, dec.sel_idx, dec.sel_cnt, dec.sel_stride)
    assert e.value.status == 1


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_gaussian_head_dim_64_and_an_empty_request(alpha):
    """D = 64, and a batch whose first request holds no tokens: that request
    selects nothing (count 0, tau_hat NaN) and its output is 0; the others
    match the oracle."""
    cfg = config(3, small=True).replace(D=64, len_range=(40, 700))
    wl = make_workload(cfg)
    c = wl.cfg
    dec = make_decoder(wl, extra=dict(gaussian=True, alpha=alpha))
    lens = dec.seq_lens.clone()
    dec.seq_lens[0] = 0                                     # an empty request
    q = dev_bits(wl.q(0), c.dtype)
    dec.attend(q)
    torch.cuda.synchronize()
    assert int(dec.sel_cnt[0].abs().sum()) == 0
    assert torch.isnan(dec.tau_hat[0]).all()
    assert torch.all(dec.out[0].float() == 0)
    heads = [(b, g) for b in range(1, c.B) for g in range(c.H_q)]
    assert _check_selection(dec, wl, 0, wl.q(0), alpha, heads) >= 0.9 * len(heads)
    sel = dec.sel_idx.cpu().numpy()
    cnt = dec.sel_cnt.cpu().numpy()
    out = dec.out.float().cpu().numpy()
    sc = _scale(c)
    for b, gq in heads:
        h = gq // c.G
        L = int(wl.prefill_lens[b])
        pos = O.selected_positions(sel[b, gq, :cnt[b, gq]], L, c.ps)
        k = O.decode_kdt(wl.k_seq(b)[:, h, :][pos], c.dtype)
        v = O.decode_kdt(wl.v_seq(b)[:, h, :][pos], c.dtype)
        o, _, _ = O.attention_entmax(O.decode_kdt(wl.q(0)[b, gq], c.dtype)[None], k, v, sc, alpha)
        assert_attention(out[b, gq][None], o)
    dec.seq_lens.copy_(lens)
    assert dev_status(dec) == 0


@pytest.mark.parametrize("H_q,H_kv", [(32, 2), (2, 2), (12, 2)])
def test_gaussian_query_groups(H_q, H_kv):
    """Groups of 16, 1 and 6 query heads per KV head (the moments' two tile
    shapes, empty rows of a tile): moments, tau_hat, selection and attention
    against the oracle."""
    wl, dec = _gauss_decoder(5, 1.5, H_q=H_q, H_kv=H_kv)
    c = wl.cfg
    q = dev_bits(wl.q(0), c.dtype)
    dec.attend(q)
    torch.cuda.synchronize()
    heads = [(b, g) for b in range(c.B) for g in range(c.H_q)]
    assert _check_selection(dec, wl, 0, wl.q(0), 1.5, heads) >= 0.9 * len(heads)
    sel = dec.sel_idx.cpu().numpy()
    cnt = dec.sel_cnt.cpu().numpy()
    out = dec.out.float().cpu().numpy()
    sc = _scale(c)
    for b, gq in heads:
        h = gq // c.G
        L = int(wl.prefill_lens[b])
        pos = O.selected_positions(sel[b, gq, :cnt[b, gq]], L, c.ps)
        k = O.decode_kdt(wl.k_seq(b)[:, h, :][pos], c.dtype)
        v = O.decode_kdt(wl.v_seq(b)[:, h, :][pos], c.dtype)
        o, _, _ = O.attention_entmax(O.decode_kdt(wl.q(0)[b, gq], c.dtype)[None], k, v, sc, 1.5)
        assert_attention(out[b, gq][None], o)
    assert dev_status(dec) == 0


def test_gauss_select_bad_block_and_overflow():
    """A page with an out-of-range block id gets (-inf, 0) moments, is never
    kept and sets SA_DEV_BAD_BLOCK, the other pages' moments unchanged; a
    request longer than its block-table row sets SA_DEV_OVERFLOW and is read
    up to the row's end (selection ascending, ending at the row's last page);
    the untouched request still matches the oracle."""
    from sparse_paged_kv_page_gb300 import sa_gauss_select
    from sparse_paged_kv_page_gb300._lib import SA_DEV_BAD_BLOCK, SA_DEV_OVERFLOW
    wl, dec = _gauss_decoder(3)
    c = wl.cfg
    q = dev_bits(wl.q(0), c.dtype)
    n1 = O.num_pages(int(wl.prefill_lens[1]), c.ps)
    assert n1 >= 3
    lens = dec.seq_lens.clone()
    bt = dec.block_table.clone()
    dec.block_table[1, 1] = wl.num_blocks + 5               # page 1 of request 1 (never its tail)
    dec.seq_lens[0] = dec.block_table.shape[1] * c.ps + 100  # more pages than the row holds
    sa_gauss_select(dec.cache.struct, dec.batch, q, c.H_q, 1.5, dec.scale, dec.moments, dec.max_pages,
                    dec.sel_idx, dec.sel_cnt, dec.sel_stride, tau_hat=dec.tau_hat,
                    dev_status=dec.dev_status)
    torch.cuda.synchronize()
    st = dev_status(dec)
    assert st & SA_DEV_BAD_BLOCK and st & SA_DEV_OVERFLOW
    mom = dec.moments.cpu().numpy()
    sel = dec.sel_idx.cpu().numpy()
    cnt = dec.sel_cnt.cpu().numpy()
    row = dec.block_table.shape[1]
    for g in range(c.H_q):
        assert mom[1, g, 1, 0] == -np.inf and mom[1, g, 1, 1] == 0.0
        assert 1 not in sel[1, g, :cnt[1, g]]
        r = _oracle_head(wl, 1, g, 0, wl.q(0), 1.5)
        m = mom[1, g, :n1, 0].astype(np.float64)
        keep = np.arange(n1) != 1
        qd = np.abs(O.decode_kdt(wl.q(0)[1, g], c.dtype))
        tol_m = 1e-5 * _scale(c) * (np.abs(r["mean"]) @ qd) + 1e-9
        assert np.all(np.abs(m - r["m"])[keep] <= tol_m[keep])
        s0 = sel[0, g, :cnt[0, g]]
        assert 1 <= cnt[0, g] <= row and s0[-1] == row - 1 and np.all(np.diff(s0) > 0)
    assert _check_selection(dec, wl, 0, wl.q(0), 1.5, [(2, g) for g in range(c.H_q)]) >= 0
    dec.block_table.copy_(bt)
    dec.seq_lens.copy_(lens)
