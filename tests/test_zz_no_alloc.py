"""The allocation-free decode entry point, for callers that cannot allocate
device memory at the call site (plugins given fixed buffers, frozen memory
plans, allocation-free real-time loops).

It must give the same results as sa_sparse_decode with a caller workspace and
as the oracle's attention over the same given selection -- within the decode
tolerance of the other tests -- on two calls in a row (the second reuses the
shared scratch the first left behind), and refuse sizes that need more scratch
than its fixed capacity. Kept in a file collected last.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import make_decoder, dev_bits, assert_attention

pytestmark = pytest.mark.gpu


def _selection(wl, k, seed):
    c = wl.cfg
    rng = np.random.default_rng(seed)
    sel = np.zeros((c.B, c.H_kv, k), dtype=np.int32)
    cnt = np.zeros((c.B, c.H_kv), dtype=np.int32)
    for b in range(c.B):
        n = -(-int(wl.prefill_lens[b]) // c.ps)
        for h in range(c.H_kv):
            m = min(k, n)
            sel[b, h, :m] = np.sort(rng.choice(n, size=m, replace=False))
            cnt[b, h] = m
    return torch.from_numpy(sel).cuda(), torch.from_numpy(cnt).cuda()


def test_noalloc_matches_workspace_decode_twice():
    import sparse_paged_kv_page_gb300 as S
    cfg = config(5, small=True)
    wl = make_workload(cfg)
    dec = make_decoder(wl, stale="nan")
    sel, cnt = _selection(wl, cfg.topk, 3)
    q = dev_bits(wl.q(0), cfg.dtype)
    ws = S.alloc_decode_workspace(cfg.B, cfg.H_kv, cfg.H_q, cfg.D, cfg.ps, cfg.topk)
    assert S.sa_decode_workspace_size(cfg.B, cfg.H_kv, cfg.H_q, cfg.D, cfg.ps, cfg.topk) > 4 * cfg.B * cfg.H_kv
    ref_o = torch.empty_like(dec.out)
    ref_l = torch.empty_like(dec.lse)
    S.sa_sparse_decode(dec.cache.struct, dec.batch, q, cfg.H_q, sel, cnt, cfg.topk, 0.0, ref_o,
                       lse=ref_l, workspace=ws, dev_status=dec.dev_status)
    # the oracle's attention of every (request, KV head) over the same given selection
    sc = O.default_scale(cfg.D)
    sel_h, cnt_h = sel.cpu().numpy(), cnt.cpu().numpy()
    want = {}
    for b in range(cfg.B):
        L = int(wl.prefill_lens[b])
        for h in range(cfg.H_kv):
            pos = O.selected_positions(sel_h[b, h, :cnt_h[b, h]], L, cfg.ps)
            k = O.decode_kdt(wl.k_seq(b, head=h)[pos], cfg.dtype)
            v = O.decode_kdt(wl.v_seq(b, head=h)[pos], cfg.dtype)
            qg = O.decode_kdt(wl.q(0)[b, h * cfg.G:(h + 1) * cfg.G], cfg.dtype)
            want[(b, h)] = O.attention(qg, k, v, sc)[:2]
    for call in range(2):
        out = torch.full_like(dec.out, float("nan"))
        lse = torch.full_like(dec.lse, float("nan"))
        S.sa_sparse_decode_noalloc(dec.cache.struct, dec.batch, q, cfg.H_q, sel, cnt, cfg.topk, 0.0,
                                   out, lse=lse, dev_status=dec.dev_status)
        torch.cuda.synchronize()
        a, b = out.float().cpu().numpy(), ref_o.float().cpu().numpy()
        assert np.all(np.abs(a - b) <= 2e-2 + 2e-2 * np.abs(b)), call
        assert np.allclose(lse.cpu().numpy(), ref_l.cpu().numpy(), atol=1e-3), call
        ln = lse.cpu().numpy()
        for (bb, h), (wo, wlse) in want.items():
            rows = slice(h * cfg.G, (h + 1) * cfg.G)
            assert_attention(a[bb, rows], wo, ln[bb, rows], wlse)
    assert int(dec.dev_status.item()) == 0


def test_noalloc_rejects_more_than_its_capacity():
    import sparse_paged_kv_page_gb300 as S
    cap = S.sa_sparse_decode_noalloc_capacity()
    # token-level shapes with a very long selection need more scratch than the array holds
    B, H, Hq, D, ps, stride = 1, 8, 128, 128, 1, 1 << 20
    assert S.sa_decode_workspace_size(B, H, Hq, D, ps, stride) > cap
    k = torch.zeros((4, H, ps, D), dtype=torch.bfloat16, device="cuda")
    cache = S.make_cache(k, k.clone(), None)
    batch = S.make_batch(torch.zeros((B, 4), dtype=torch.int32, device="cuda"),
                         torch.zeros((B,), dtype=torch.int32, device="cuda"))
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    sel = torch.zeros((B, H, stride), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B, H), dtype=torch.int32, device="cuda")
    out = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(S.SaError) as e:
        S.sa_sparse_decode_noalloc(cache, batch, q, Hq, sel, cnt, stride, 0.0, out)
    assert e.value.status == 3          # SA_ERR_WORKSPACE, nothing launched
