"""sa_sparse_decode on the GPU against the oracle's float64 attention.

Selections come from the generator (random page subsets, any order), so the
decode kernel is compared on exactly the oracle's inputs: outputs within
atol 2e-2 + rtol 2e-2 (bf16/fp16 I/O), lse within 1e-3, logits within 1e-4
relative. Also: all pages = dense attention, empty and ragged selections,
NaN-poisoned stale slots, and bit-identical results across block tables.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload, reverse_interleaved, shuffled_table, contiguous_table
from gpu_util import (make_decoder, dev_bits, dev_status, host_bits, assert_attention, TDT)

pytestmark = pytest.mark.gpu


def _decode(dec, q, sel_np, cnt_np, stride, logits=False):
    from sparse_paged_kv_page_gb300 import sa_sparse_decode, alloc_decode_workspace
    B, H = cnt_np.shape
    sel = torch.from_numpy(sel_np.astype(np.int32)).cuda()
    cnt = torch.from_numpy(cnt_np.astype(np.int32)).cuda()
    out = torch.full((B, dec.H_q, dec.D), float("nan"), dtype=dec.dtype, device="cuda")
    lse = torch.full((B, dec.H_q), float("nan"), dtype=torch.float32, device="cuda")
    ws = alloc_decode_workspace(B, H, dec.H_q, dec.D, dec.ps, stride)
    lg = None
    if logits:
        lg = torch.full((B, dec.H_q, stride * dec.ps), float("nan"), device="cuda")
    sa_sparse_decode(dec.cache.struct, dec.batch, q, dec.H_q, sel, cnt, stride, dec.scale, out,
                     lse=lse, logits=lg, logits_stride=stride * dec.ps if logits else 0,
                     workspace=ws, dev_status=dec.dev_status)
    torch.cuda.synchronize()
    assert int(ws[:4 * B * H].view(torch.int32).abs().sum().item()) == 0   # tickets reset
    return out, lse, lg


def _random_selection(wl, rng, k, order="asc"):
    c = wl.cfg
    sel = np.full((c.B, c.H_kv, k), -1, dtype=np.int64)
    cnt = np.zeros((c.B, c.H_kv), dtype=np.int64)
    for b in range(c.B):
        n = O.num_pages(wl.prefill_lens[b], c.ps)
        for h in range(c.H_kv):
            m = min(k, n) if n else 0
            if m and rng.random() < 0.15:
                m = int(rng.integers(0, m + 1))
            pick = rng.choice(n, size=m, replace=False) if m else np.zeros(0, dtype=np.int64)
            if order == "asc":
                pick = np.sort(pick)
            sel[b, h, :m] = pick
            cnt[b, h] = m
    return sel, cnt


def _check(dec, wl, q_bits, sel, cnt, out, lse, lg=None):
    c = wl.cfg
    o_np = out.float().cpu().numpy()
    l_np = lse.cpu().numpy()
    lg_np = lg.cpu().numpy() if lg is not None else None
    sc = c.scale if c.scale > 0 else O.default_scale(c.D)
    for b in range(c.B):
        L = int(wl.prefill_lens[b])
        for h in range(c.H_kv):
            m = int(cnt[b, h])
            pos = O.selected_positions(sel[b, h, :m], L, c.ps)
            ks = wl.k_seq(b)[:, h, :]
            vs = wl.v_seq(b)[:, h, :]
            q = O.decode_kdt(q_bits[b, h * c.G:(h + 1) * c.G], c.dtype)
            o, ls, z = O.attention(q, O.decode_kdt(ks[pos], c.dtype), O.decode_kdt(vs[pos], c.dtype), sc)
            assert_attention(o_np[b, h * c.G:(h + 1) * c.G], o, l_np[b, h * c.G:(h + 1) * c.G], ls)
            if lg_np is not None:
                # selection token i = entry * ps + slot; invalid slots are -inf
                got = lg_np[b, h * c.G:(h + 1) * c.G, :m * c.ps]
                want = np.full_like(got, -np.inf, dtype=np.float64)
                j = 0
                for e in range(m):
                    p = int(sel[b, h, e])
                    f = min(c.ps, L - p * c.ps)
                    want[:, e * c.ps:e * c.ps + f] = z[:, j:j + f]
                    j += f
                fin = np.isfinite(want)
                assert np.array_equal(np.isfinite(got), fin)
                assert np.all(np.abs(got[fin] - want[fin]) <= 1e-4 * (1 + np.abs(want[fin])))


@pytest.mark.parametrize("cid", [1, 2, 3, 5])
@pytest.mark.parametrize("stale", ["normal3", "nan"])
def test_decode_random_selections(cid, stale):
    wl = make_workload(config(cid, small=True))
    dec = make_decoder(wl, stale=stale)
    rng = np.random.default_rng([cid, len(stale)])
    k = max(wl.cfg.topk, 4)
    sel, cnt = _random_selection(wl, rng, k, order="asc" if cid != 3 else "any")
    qb = wl.q(0)
    out, lse, lg = _decode(dec, dev_bits(qb, wl.cfg.dtype), sel, cnt, k, logits=True)
    _check(dec, wl, qb, sel, cnt, out, lse, lg)
    assert dev_status(dec) == 0


@pytest.mark.parametrize("G,D,dtype", [(1, 128, "bf16"), (3, 64, "fp16"), (7, 128, "bf16"),
                                       (8, 64, "bf16"), (16, 128, "fp16")])
def test_decode_group_sizes_all_pages_is_dense(G, D, dtype):
    cfg = config(3, small=True).replace(H_q=2 * G, H_kv=2, D=D, dtype=dtype, len_range=(1, 333))
    wl = make_workload(cfg)
    dec = make_decoder(wl, stale="nan")
    k = wl.max_pages
    sel = np.zeros((cfg.B, cfg.H_kv, k), dtype=np.int64)
    cnt = np.zeros((cfg.B, cfg.H_kv), dtype=np.int64)
    for b in range(cfg.B):
        n = O.num_pages(wl.prefill_lens[b], cfg.ps)
        sel[b, :, :n] = np.arange(n)
        cnt[b, :] = n
    qb = wl.q(0)
    out, lse, _ = _decode(dec, dev_bits(qb, dtype), sel, cnt, k)
    _check(dec, wl, qb, sel, cnt, out, lse)


@pytest.mark.parametrize("B,topk", [(1, 64), (1, 3), (2, 48), (12, 64)])
def test_decode_split_counts(B, topk):
    # different (units, tiles) give different split counts; all must equal single-shot
    cfg = config(5, small=True).replace(B=B, prefill=(1500,) * B, topk=topk, num_blocks=None)
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    rng = np.random.default_rng([B, topk])
    sel, cnt = _random_selection(wl, rng, topk)
    qb = wl.q(0)
    out, lse, _ = _decode(dec, dev_bits(qb, cfg.dtype), sel, cnt, topk)
    _check(dec, wl, qb, sel, cnt, out, lse)


@pytest.mark.parametrize("topk", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("G,D,dtype", [(8, 128, "bf16"), (3, 64, "fp16"), (16, 128, "bf16")])
def test_decode_every_cluster_size(topk, G, D, dtype):
    # One request with two KV heads, a selection of topk pages of 16 tokens
    # (one tile each): the split count is min(8, topk) on any GPU of 8 or more
    # SMs, so every cluster size of the split merge runs, with output slices
    # of G * D that do not always divide evenly, and some units selecting
    # fewer pages than splits (empty partials)
    cfg = config(5, small=True).replace(B=1, H_q=2 * G, H_kv=2, D=D, dtype=dtype,
                                        prefill=(1500,), topk=topk, num_blocks=None)
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    rng = np.random.default_rng([topk, G, D])
    sel, cnt = _random_selection(wl, rng, topk)
    qb = wl.q(0)
    out, lse, _ = _decode(dec, dev_bits(qb, dtype), sel, cnt, topk)
    _check(dec, wl, qb, sel, cnt, out, lse)
    assert dev_status(dec) == 0


def test_empty_and_zero_length():
    cfg = config(3, small=True).replace(B=3, len_range=(1, 50))
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    sl = dec.seq_lens.clone()
    dec.seq_lens[2] = 0                               # a request with no tokens
    sel = np.zeros((3, cfg.H_kv, 4), dtype=np.int64)
    cnt = np.array([[0, 1], [2, 0], [1, 1]])
    out, lse, _ = _decode(dec, dev_bits(wl.q(0), cfg.dtype), sel, cnt, 4)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    G = cfg.G
    for b, h in [(0, 0), (1, 1), (2, 0), (2, 1)]:
        assert np.all(o[b, h * G:(h + 1) * G] == 0) and np.all(l[b, h * G:(h + 1) * G] == -np.inf)
    assert dev_status(dec) & 1                        # page 0 of an empty request is out of range
    dec.seq_lens.copy_(sl)


@pytest.mark.parametrize("table", ["reverse", "shuffle", "contiguous"])
def test_block_tables_give_bit_identical_results(table):
    cfg = config(5, small=True).replace(table=table)
    wl = make_workload(cfg)
    dec = make_decoder(wl, stale="nan")
    rng = np.random.default_rng(3)
    sel, cnt = _random_selection(wl, rng, cfg.topk)
    out, lse, _ = _decode(dec, dev_bits(wl.q(0), cfg.dtype), sel, cnt, cfg.topk)
    ref_cfg = cfg.replace(table="contiguous")
    wl2 = make_workload(ref_cfg)
    dec2 = make_decoder(wl2, stale="normal3")
    out2, lse2, _ = _decode(dec2, dev_bits(wl2.q(0), cfg.dtype), sel, cnt, cfg.topk)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)
    _check(dec, wl, wl.q(0), sel, cnt, out, lse)


def test_token_level_rows_and_logits():
    wl = make_workload(config(4, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    rng = np.random.default_rng(9)
    k = 120
    sel = np.zeros((c.B, c.H_kv, k), dtype=np.int64)
    cnt = np.zeros((c.B, c.H_kv), dtype=np.int64)
    for b in range(c.B):
        for h in range(c.H_kv):
            m = int(rng.integers(1, k + 1))
            sel[b, h, :m] = np.sort(rng.choice(int(wl.prefill_lens[b]), size=m, replace=False))
            cnt[b, h] = m
    qb = wl.q(0)
    out, lse, lg = _decode(dec, dev_bits(qb, c.dtype), sel, cnt, k, logits=True)
    _check(dec, wl, qb, sel, cnt, out, lse, lg)
