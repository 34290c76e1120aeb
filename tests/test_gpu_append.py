"""sa_append_kv on the GPU against the oracle: pool contents, page statistics,
H2O slot reset and retained-list appends. Inputs from sa_synth, expected values
from oracle/ (page statistics over the logical key sequence)."""
import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden
from sa_synth import config, make_workload, Config
from gpu_util import dev_bits, host_bits, make_decoder, step_inputs, dev_status, TDT

pytestmark = pytest.mark.gpu


def _meta_of_block(dec, blk, h):
    m = host_bits(dec.cache.meta[blk, h])                      # [3, D] bits
    return [O.decode_kdt(m[i], dec_dtype(dec)) for i in range(3)]


def dec_dtype(dec):
    return "bf16" if dec.dtype == torch.bfloat16 else "fp16"


def _check_request_meta(dec, wl, b, steps_done, pages=None):
    c = wl.cfg
    L = wl.seq_len(b, steps_done)
    mn, mx, me = O.cache_meta(wl.k_seq(b, steps_done), L, c.ps, c.dtype)
    meta = host_bits(dec.cache.meta)                          # [NB, H, 3, D]
    n = O.num_pages(L, c.ps)
    for p in (range(n) if pages is None else pages):
        blk = int(wl.block_table[b, p])
        for h in range(c.H_kv):
            got = [O.decode_kdt(meta[blk, h, i], c.dtype) for i in range(3)]
            assert np.array_equal(got[0], mn[p, h]), (b, p, h, "min")
            assert np.array_equal(got[1], mx[p, h]), (b, p, h, "max")
            assert np.array_equal(got[2], me[p, h]), (b, p, h, "mean")


def _check_request_rows(dec, wl, b, steps_done):
    c = wl.cfg
    L = wl.seq_len(b, steps_done)
    pos = np.arange(L)
    kp, vp = host_bits(dec.cache.k), host_bits(dec.cache.v)
    ks, vs = wl.k_seq(b, steps_done), wl.v_seq(b, steps_done)
    for h in range(c.H_kv):
        assert np.array_equal(O.gather_rows(kp, wl.block_table[b], pos, h, c.ps), ks[:, h])
        assert np.array_equal(O.gather_rows(vp, wl.block_table[b], pos, h, c.ps), vs[:, h])


@pytest.mark.parametrize("cid", [1, 3, 5])
@pytest.mark.parametrize("stale", ["normal3", "nan"])
def test_prefill_rows_and_meta(cid, stale):
    wl = make_workload(config(cid, small=True))
    dec = make_decoder(wl, stale=stale)
    assert dev_status(dec) == 0
    assert dec.seq_lens.cpu().tolist() == wl.prefill_lens.tolist()
    for b in range(wl.cfg.B):
        _check_request_rows(dec, wl, b, 0)
        _check_request_meta(dec, wl, b, 0)
    # blocks no request references keep their stale contents
    used = set()
    for b in range(wl.cfg.B):
        used.update(wl.block_table[b, :O.num_pages(wl.prefill_lens[b], wl.cfg.ps)].tolist())
    free = [x for x in range(wl.num_blocks) if x not in used][:8]
    if free and stale == "nan":
        assert torch.isnan(dec.cache.k[free].float()).all()


@pytest.mark.parametrize("dtype,D,G", [("fp16", 128, 4), ("bf16", 64, 3), ("fp16", 64, 8)])
def test_decode_appends_refresh_tail_page(dtype, D, G):
    cfg = config(2, small=True).replace(dtype=dtype, D=D, H_q=2 * G, H_kv=2, decode_steps=20,
                                        prefill=(37,))
    wl = make_workload(cfg)
    dec = make_decoder(wl, stale="nan")
    for t in range(cfg.decode_steps):
        _, kn, vn = step_inputs(wl, t)
        dec.append(kn, vn)
        torch.cuda.synchronize()
        L = wl.seq_len(0, t + 1)
        _check_request_meta(dec, wl, 0, t + 1, pages=[(L - 1) // cfg.ps])
    assert dev_status(dec) == 0
    _check_request_rows(dec, wl, 0, cfg.decode_steps)
    _check_request_meta(dec, wl, 0, cfg.decode_steps)


def test_ragged_multi_request_prefill_and_appends():
    cfg = config(3, small=True).replace(len_range=(1, 90), B=5)
    wl = make_workload(cfg, extra_steps=6)
    dec = make_decoder(wl, stale="nan")
    for t in range(6):
        _, kn, vn = step_inputs(wl, t)
        dec.append(kn, vn)
    torch.cuda.synchronize()
    for b in range(cfg.B):
        _check_request_rows(dec, wl, b, 6)
        _check_request_meta(dec, wl, b, 6)
    assert dev_status(dec) == 0


def test_fill_resets_exactly_the_written_slots():
    # vortex_torch PR 6, "Fill(0.0) resets hh_score for exactly the pages written":
    # 64 slots prefilled 7.5, tokens written to slots {3, 5, 11, 40}.
    g = golden("vortex_h2o_constants.txt")
    nslots = int(g["fill_num_pages"])
    touched = [int(x) for x in g["fill_touched"].split()]
    pre = float(g["fill_prefill_value"])
    cfg = Config(cid=0, name="fill", B=1, H_q=1, H_kv=1, D=128, ps=1, dtype="bf16",
                 prefill=(len(touched),), num_blocks=nslots, table="contiguous", budget=3,
                 n_sink=1, grace=1, decay=0.984375)
    wl = make_workload(cfg)
    from sparse_paged_kv_page_gb300.step import SparseDecoder
    dec = SparseDecoder(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=128, page_size=1,
                        num_blocks=nslots, bt_stride=nslots, ret_cap=nslots, budget=3, n_sink=1,
                        grace=1, decay=0.984375)
    dec.cache.hh.fill_(pre)
    bt = torch.zeros((1, nslots), dtype=torch.int32)
    bt[0, :len(touched)] = torch.tensor(touched, dtype=torch.int32)
    dec.set_block_table(bt)
    dec.prefill(dev_bits(wl.k_pre, "bf16"), dev_bits(wl.v_pre, "bf16"), [len(touched)])
    torch.cuda.synchronize()
    hh = dec.cache.hh[:, 0].float().cpu().numpy()
    mask = np.zeros(nslots, dtype=bool)
    mask[touched] = True
    assert np.all(hh[mask] == 0.0)
    assert np.all(hh[~mask] == pre)
    assert dec.ret_cnt.item() == len(touched)
    assert dec.ret_pos[0, 0, :len(touched)].cpu().tolist() == list(range(len(touched)))


def test_token_level_prefill_appends_retained_lists():
    wl = make_workload(config(4, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    rc = dec.ret_cnt.cpu().numpy()
    rp = dec.ret_pos.cpu().numpy()
    for b in range(c.B):
        for h in range(c.H_kv):
            L = int(wl.prefill_lens[b])
            assert rc[b, h] == L and np.array_equal(rp[b, h, :L], np.arange(L))
    hh = dec.cache.hh.float().cpu().numpy()
    for b in range(c.B):
        slots = wl.block_table[b, :int(wl.prefill_lens[b])]
        assert np.all(hh[slots] == 0.0)
    assert dev_status(dec) == 0


def test_overflow_and_bad_block_are_flagged_not_faulted():
    cfg = config(1).replace(num_blocks=64)
    wl = make_workload(cfg)
    from sparse_paged_kv_page_gb300.step import SparseDecoder
    dec = SparseDecoder(batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, page_size=16,
                        num_blocks=64, bt_stride=2, topk=4)
    dec.set_block_table(torch.tensor([[63, 62]], dtype=torch.int32))
    # 40 tokens into a 2-page (32-token) table: the excess is dropped, overflow flagged
    k = dev_bits(wl.k_pre[:40], "bf16")
    dec.prefill(k, k, [40])
    torch.cuda.synchronize()
    assert dec.seq_lens.item() == 32 and dev_status(dec) & 2
    dec2 = SparseDecoder(batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, page_size=16,
                         num_blocks=64, bt_stride=4, topk=4)
    dec2.set_block_table(torch.tensor([[63, 99, 1, 2]], dtype=torch.int32))   # 99 is out of range
    dec2.prefill(k, k, [40])
    torch.cuda.synchronize()
    assert dev_status(dec2) & 1
