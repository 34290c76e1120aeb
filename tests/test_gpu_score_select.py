"""sa_score_pages and sa_select_topk on the GPU against the oracle.

Scores: within 1e-4 of the oracle's float64 plain-form scores, norm-wise.
Selection: bit-exact against the oracle's selector applied to the same
generator-drawn float32 scores (ties, signed zeros, NaN, -inf included); in the
chained path the GPU's selection must be a valid top-k for scores within the
float32 error bound of the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import (make_decoder, step_inputs, dev_status, host_bits, score_norm, assert_scores,
                      score_error_bound, assert_selection_valid)

pytestmark = pytest.mark.gpu


def _oracle_scores(wl, b, h, steps_done, q_bits):
    c = wl.cfg
    L = wl.seq_len(b, steps_done)
    mn, mx, me = O.head_meta(wl.k_seq(b, steps_done)[:, h, :], L, c.ps, c.dtype)
    q = O.decode_kdt(q_bits[h * c.G:(h + 1) * c.G], c.dtype)
    S = O.score_pages(mn, mx, me, q, c.w_avg, c.w_peak)
    return S, score_norm(mn, mx, me, q, c.w_avg, c.w_peak), L


def _run_scores(dec, wl, t):
    q, _, _ = step_inputs(wl, t)
    from sparse_paged_kv_page_gb300 import sa_score_pages, sa_select_topk
    sa_score_pages(dec.cache.struct, dec.batch, q, wl.cfg.H_q, wl.cfg.w_avg, wl.cfg.w_peak,
                   dec.scores, dec.max_pages, dev_status=dec.dev_status)
    sa_select_topk(dec.scores, dec.max_pages, dec.batch, wl.cfg.ps, wl.cfg.H_kv, wl.cfg.topk,
                   dec.sel_idx, dec.sel_cnt, dev_status=dec.dev_status)
    torch.cuda.synchronize()
    return wl.q(t)


@pytest.mark.parametrize("cid", [1, 2, 3, 5])
def test_scores_and_selection_small_configs(cid):
    wl = make_workload(config(cid, small=True))
    dec = make_decoder(wl)
    qb = _run_scores(dec, wl, 0)
    scores = dec.scores.cpu().numpy()
    sel = dec.sel_idx.cpu().numpy()
    cnt = dec.sel_cnt.cpu().numpy()
    c = wl.cfg
    for b in range(c.B):
        for h in range(c.H_kv):
            S, A, L = _oracle_scores(wl, b, h, 0, qb[b])
            n = O.num_pages(L, c.ps)
            assert_scores(scores[b, h, :n], S, A)
            assert cnt[b, h] == min(c.topk, n)
            eps = score_error_bound(A, c.D, c.G)
            assert_selection_valid(sel[b, h, :cnt[b, h]], S, eps, n, c.topk)
    assert dev_status(dec) == 0


@pytest.mark.parametrize("G", [1, 3, 4, 7, 8, 16])
@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "fp16")])
def test_scores_group_sizes(G, D, dtype):
    cfg = config(3, small=True).replace(H_q=2 * G, H_kv=2, D=D, dtype=dtype, len_range=(5, 400),
                                        w_avg=0.7, w_peak=0.3)
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    qb = _run_scores(dec, wl, 0)
    scores = dec.scores.cpu().numpy()
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            S, A, L = _oracle_scores(wl, b, h, 0, qb[b])
            assert_scores(scores[b, h, :O.num_pages(L, cfg.ps)], S, A)


@pytest.mark.parametrize("H_kv", [3, 6, 8, 12, 16])
@pytest.mark.parametrize("D", [128, 64])
def test_scores_kv_head_counts(H_kv, D):
    """Chunks gather several KV heads of a block per copy (as many as divide
    both H_kv and the lane groups): counts that split into 1, 2, 4, 8 or 16."""
    cfg = config(3, small=True).replace(H_q=2 * H_kv, H_kv=H_kv, D=D, len_range=(5, 700),
                                        w_avg=0.6, w_peak=0.4)
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    qb = _run_scores(dec, wl, 0)
    scores = dec.scores.cpu().numpy()
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            S, A, L = _oracle_scores(wl, b, h, 0, qb[b])
            assert_scores(scores[b, h, :O.num_pages(L, cfg.ps)], S, A)
    assert dev_status(dec) == 0


def _run_select(scores_np, lens, ps, topk, H):
    from sparse_paged_kv_page_gb300 import make_batch, sa_select_topk
    B, _, maxp = scores_np.shape
    sc = torch.from_numpy(scores_np.astype(np.float32)).cuda()
    bt = torch.zeros((B, maxp), dtype=torch.int32, device="cuda")
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    batch = make_batch(bt, sl)
    sel = torch.full((B, H, topk), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa_select_topk(sc, maxp, batch, ps, H, topk, sel, cnt, dev_status=st)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), cnt.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("kind", ["continuous", "ties", "specials"])
@pytest.mark.parametrize("topk", [1, 2, 7, 64, 256])
def test_select_bit_exact_on_generated_scores(kind, topk):
    rng = np.random.default_rng([77, topk, len(kind)])
    B, H, maxp, ps = 3, 4, 3000, 16
    if kind == "continuous":
        s = rng.standard_normal((B, H, maxp)).astype(np.float32)
    elif kind == "ties":
        s = rng.integers(-3, 4, size=(B, H, maxp)).astype(np.float32) * 0.5
    else:
        pool = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-30, -1e-30, 3.0],
                        dtype=np.float32)
        s = rng.choice(pool, size=(B, H, maxp))
    lens = [maxp * ps, int(rng.integers(1, 200)) * ps - 3, 0]
    sel, cnt, st = _run_select(s, lens, ps, topk, H)
    assert st == 0
    for b in range(B):
        n = O.num_pages(lens[b], ps)
        for h in range(H):
            want = O.select_pages(s[b, h], n, topk)
            assert cnt[b, h] == len(want)
            assert np.array_equal(sel[b, h, :cnt[b, h]], want), (b, h)
            assert np.all(sel[b, h, cnt[b, h]:] == -7)


@pytest.mark.parametrize("kind", ["boundary_ties", "narrow", "outlier"])
@pytest.mark.parametrize("topk", [8, 256])
def test_select_adversarial_rows(kind, topk):
    """Rows that stress the radix select's digits: exact duplicates of the
    boundary score scattered over the row (the kept ones are the lowest page
    indices among them), a spread of only ~1e-6 (keys that differ in their
    low mantissa bits alone, so every digit is needed), and one huge outlier
    (the first digit puts it alone above all other keys)."""
    rng = np.random.default_rng([13, topk, len(kind)])
    B, H, maxp, ps = 2, 3, 9000, 16
    s = rng.standard_normal((B, H, maxp)).astype(np.float32)
    if kind == "boundary_ties":
        for b in range(B):
            for h in range(H):
                row = s[b, h, :maxp - 1]
                kth = np.sort(row)[::-1][topk - 2] if topk > 1 else row.max()
                row[rng.choice(maxp - 1, size=40, replace=False)] = kth
    elif kind == "narrow":
        s = (1.0 + 1e-6 * s).astype(np.float32)
    else:
        s[:, :, 17] = 3e38
    lens = [maxp * ps, (maxp - 333) * ps + 1]
    sel, cnt, st = _run_select(s, lens, ps, topk, H)
    assert st == 0
    for b in range(B):
        n = O.num_pages(lens[b], ps)
        for h in range(H):
            assert np.array_equal(sel[b, h, :cnt[b, h]], O.select_pages(s[b, h], n, topk)), (b, h)


@pytest.mark.parametrize("maxp", [2048, 2049, 8192, 9000, 16384, 16385])
def test_select_row_lengths(maxp):
    """Rows of up to 16 K pages keep their keys in registers (2, 4, 8 or 16 per
    thread); longer rows in shared memory: both sides of every boundary."""
    rng = np.random.default_rng([91, maxp])
    B, H, ps = 2, 2, 16
    s = rng.standard_normal((B, H, maxp)).astype(np.float32)
    s[1, 1] = np.round(s[1, 1] * 2) / 2                      # heavy ties
    lens = [maxp * ps, (maxp - 700) * ps + 5]
    sel, cnt, st = _run_select(s, lens, ps, 256, H)
    assert st == 0
    for b in range(B):
        n = O.num_pages(lens[b], ps)
        for h in range(H):
            assert np.array_equal(sel[b, h, :cnt[b, h]], O.select_pages(s[b, h], n, 256)), (b, h)


@pytest.mark.parametrize("bos,eos", [(0, 1), (2, 1), (4, 8), (1, 3)])
@pytest.mark.parametrize("kind", ["continuous", "ties", "specials"])
@pytest.mark.parametrize("topk", [12, 64, 256])
def test_select_reserved_bit_exact(bos, eos, kind, topk):
    """Reserved leading / trailing pages (the vortex windows): reserved pages
    kept, top-k over the window between them, against the oracle."""
    from sparse_paged_kv_page_gb300 import make_batch, sa_select_topk_reserved
    rng = np.random.default_rng([5, bos, eos, topk, len(kind)])
    B, H, maxp, ps = 3, 4, 3000, 16
    if kind == "continuous":
        s = rng.standard_normal((B, H, maxp)).astype(np.float32)
    elif kind == "ties":
        s = rng.integers(-3, 4, size=(B, H, maxp)).astype(np.float32) * 0.5
    else:
        pool = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-30, 3.0], dtype=np.float32)
        s = rng.choice(pool, size=(B, H, maxp))
    lens = [maxp * ps, (topk + 3) * ps - 7, (topk - 1) * ps]    # long, just above, below the budget
    sc = torch.from_numpy(s).cuda()
    bt = torch.zeros((B, maxp), dtype=torch.int32, device="cuda")
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sel = torch.full((B, H, topk), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, H), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa_select_topk_reserved(sc, maxp, make_batch(bt, sl), ps, H, topk, bos, eos, sel, cnt, dev_status=st)
    torch.cuda.synchronize()
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    assert int(st.item()) == 0
    for b in range(B):
        n = O.num_pages(lens[b], ps)
        for h in range(H):
            want = O.select_pages_reserved(s[b, h], n, topk, bos, eos)
            assert cnt[b, h] == len(want)
            assert np.array_equal(sel[b, h, :cnt[b, h]], want), (b, h)


def test_select_reserved_rejects_bad_windows():
    from sparse_paged_kv_page_gb300 import SaError, make_batch, sa_select_topk_reserved
    sc = torch.zeros((1, 1, 64), device="cuda")
    batch = make_batch(torch.zeros((1, 64), dtype=torch.int32, device="cuda"),
                       torch.full((1,), 64 * 16, dtype=torch.int32, device="cuda"))
    sel = torch.zeros((1, 1, 8), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    for bos, eos in [(0, 0), (-1, 1), (4, 5)]:
        with pytest.raises(SaError) as e:
            sa_select_topk_reserved(sc, 64, batch, 16, 1, 8, bos, eos, sel, cnt)
        assert e.value.status == 1


def test_select_large_candidate_count():
    rng = np.random.default_rng(5)
    B, H, maxp, ps = 1, 2, 45056, 16
    s = rng.standard_normal((B, H, maxp)).astype(np.float32)
    s[0, 1, 100:5000] = 0.25                          # a huge tie block at the boundary
    sel, cnt, st = _run_select(s, [maxp * ps], ps, 3000, H)
    for h in range(H):
        assert np.array_equal(sel[0, h, :cnt[0, h]], O.select_pages(s[0, h], maxp, 3000))


def test_bad_block_scores_nan_and_flags():
    wl = make_workload(config(1))
    dec = make_decoder(wl)
    bt = torch.from_numpy(wl.block_table.copy())
    bt[0, 3] = 1000                                   # out of range
    dec.set_block_table(bt)
    _run_scores(dec, wl, 0)
    assert dev_status(dec) & 1
    assert torch.isnan(dec.scores[0, 0, 3])
