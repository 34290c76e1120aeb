"""sa_sparse_decode_entmax on the GPU against the oracle's float64 alpha-entmax
attention ("EntmaxKV" README, How it works / Quick start).

Per (request, query head), on random page selections of the generator's
caches:
  * logits within 1e-4 relative of the oracle's (as sa_sparse_decode);
  * tau equal to the oracle's threshold of the GPU's own logits (the
    threshold is a function of the logits alone: the same support, tau within
    float32 rounding);
  * outputs within the attention tolerance (atol 2e-2, rtol 2e-2) of the
    oracle from the cache contents, and within bf16 rounding of the oracle's
    entmax of the GPU's own logits.
Plus: a support of one token returns that token's V row bit for bit, empty
selections give 0 and NaN, NaN-poisoned stale slots are never read, and bad
arguments are rejected before anything launches.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import make_decoder, dev_bits, dev_status, host_bits, assert_attention

pytestmark = pytest.mark.gpu


def _scale(c):
    return c.scale if c.scale > 0 else O.default_scale(c.D)


def _selection(wl, rng, k):
    c = wl.cfg
    sel = np.full((c.B, c.H_kv, k), -1, dtype=np.int64)
    cnt = np.zeros((c.B, c.H_kv), dtype=np.int64)
    for b in range(c.B):
        n = O.num_pages(wl.prefill_lens[b], c.ps)
        for h in range(c.H_kv):
            m = min(k, n)
            if m and rng.random() < 0.2:
                m = int(rng.integers(1, m + 1))
            pick = rng.choice(n - 1, size=m - 1, replace=False) if m > 1 else np.zeros(0, np.int64)
            pick = np.sort(np.append(pick, n - 1))           # the tail page, partly filled
            sel[b, h, :m] = pick
            cnt[b, h] = m
    return sel, cnt


def _run(dec, q, sel_np, cnt_np, stride, alpha, scale=None):
    from sparse_paged_kv_page_gb300 import sa_sparse_decode_entmax, alloc_entmax_workspace
    B, H = cnt_np.shape
    sel = torch.from_numpy(sel_np.astype(np.int32)).cuda()
    cnt = torch.from_numpy(cnt_np.astype(np.int32)).cuda()
    out = torch.full((B, dec.H_q, dec.D), float("nan"), dtype=dec.dtype, device="cuda")
    tau = torch.full((B, dec.H_q), 123.0, device="cuda")
    lg = torch.full((B, dec.H_q, stride * dec.ps), float("nan"), device="cuda")
    ws = alloc_entmax_workspace(B, H, dec.H_q, dec.D, dec.ps, stride)
    sa_sparse_decode_entmax(dec.cache.struct, dec.batch, q, dec.H_q, sel, cnt, stride, alpha,
                            dec.scale if scale is None else scale, out, tau=tau, logits=lg,
                            logits_stride=stride * dec.ps, workspace=ws, dev_status=dec.dev_status)
    torch.cuda.synchronize()
    return out, tau, lg


def _check(wl, q_bits, sel, cnt, out, tau, lg, alpha, scale):
    c = wl.cfg
    o_np = out.float().cpu().numpy()
    t_np = tau.cpu().numpy()
    lg_np = lg.cpu().numpy()
    for b in range(c.B):
        L = int(wl.prefill_lens[b])
        for h in range(c.H_kv):
            m = int(cnt[b, h])
            pos = O.selected_positions(sel[b, h, :m], L, c.ps)
            ks = O.decode_kdt(wl.k_seq(b)[:, h, :][pos], c.dtype)
            vs = O.decode_kdt(wl.v_seq(b)[:, h, :][pos], c.dtype)
            rows = slice(h * c.G, (h + 1) * c.G)
            q = O.decode_kdt(q_bits[b, rows], c.dtype)
            o, t, z = O.attention_entmax(q, ks, vs, scale, alpha)
            assert_attention(o_np[b, rows], o)
            # the GPU's logits, in selection order, at the valid slots
            got = lg_np[b, rows, :m * c.ps]
            valid = np.zeros(m * c.ps, dtype=bool)
            for e in range(m):
                f = min(c.ps, L - int(sel[b, h, e]) * c.ps)
                valid[e * c.ps:e * c.ps + f] = True
            assert np.all(got[:, ~valid] == -np.inf)
            zg = got[:, valid].astype(np.float64)
            assert np.all(np.abs(zg - z) <= 1e-4 * (1 + np.abs(z)))
            for gi in range(c.G):
                if zg.shape[1] == 0:
                    assert np.isnan(t_np[b, h * c.G + gi]) and np.all(o_np[b, h * c.G + gi] == 0)
                    continue
                # tau and the output against the oracle of the GPU's own logits
                tz = O.entmax_threshold(zg[gi], alpha)
                tg = float(t_np[b, h * c.G + gi])
                tol = (1e-6 if alpha in (1.5, 2.0) else 1e-5) * (1 + abs(tz))
                assert abs(tg - tz) <= tol, (b, h, gi, tg, tz)
                ot = O.entmax(zg[gi], alpha) @ vs
                err = np.abs(o_np[b, h * c.G + gi] - ot)
                assert np.all(err <= 2.0 ** -8 * np.abs(ot) + 1e-3), (b, h, gi, err.max())


@pytest.mark.parametrize("cid", [1, 2, 5])
@pytest.mark.parametrize("alpha", [1.5, 2.0, 1.25])
def test_entmax_random_selections(cid, alpha):
    wl = make_workload(config(cid, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    rng = np.random.default_rng([cid, int(alpha * 100)])
    k = max(c.topk, 4)
    sel, cnt = _selection(wl, rng, k)
    qb = wl.q(0)
    out, tau, lg = _run(dec, dev_bits(qb, c.dtype), sel, cnt, k, alpha)
    _check(wl, qb, sel, cnt, out, tau, lg, alpha, _scale(c))
    assert dev_status(dec) == 0


@pytest.mark.parametrize("D,G,dtype", [(64, 1, "bf16"), (128, 16, "bf16"), (128, 2, "fp16")])
def test_entmax_group_sizes(D, G, dtype):
    cfg = config(3, small=True).replace(H_kv=2, H_q=2 * G, D=D, dtype=dtype, len_range=(1, 333))
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    c = wl.cfg
    rng = np.random.default_rng(G)
    sel, cnt = _selection(wl, rng, 12)
    qb = wl.q(0)
    out, tau, lg = _run(dec, dev_bits(qb, c.dtype), sel, cnt, 12, 1.5)
    _check(wl, qb, sel, cnt, out, tau, lg, 1.5, _scale(c))
    assert dev_status(dec) == 0


@pytest.mark.parametrize("splits", [2, 3, 5, 6, 7, 8])
@pytest.mark.parametrize("G,D,dtype", [(8, 128, "bf16"), (3, 64, "fp16")])
def test_entmax_every_cluster_size(splits, G, D, dtype):
    # One request with two KV heads and a selection of 8 * splits pages of 16
    # tokens: the weighted-V pass takes min(8, tokens / 128) = splits splits
    # on any GPU of 8 or more SMs, so every cluster size of its merge runs
    k = 8 * splits
    cfg = config(5, small=True).replace(B=1, H_q=2 * G, H_kv=2, D=D, dtype=dtype,
                                        prefill=(1500,), topk=k, num_blocks=None)
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    c = wl.cfg
    rng = np.random.default_rng([splits, G, D])
    sel, cnt = _selection(wl, rng, k)
    qb = wl.q(0)
    out, tau, lg = _run(dec, dev_bits(qb, c.dtype), sel, cnt, k, 1.5)
    _check(wl, qb, sel, cnt, out, tau, lg, 1.5, _scale(c))
    assert dev_status(dec) == 0


def test_nan_stale_slots_are_never_read():
    wl = make_workload(config(2, small=True))
    dec = make_decoder(wl, stale="nan")
    c = wl.cfg
    sel, cnt = _selection(wl, np.random.default_rng(3), c.topk)
    qb = wl.q(0)
    for alpha in (1.5, 2.0):
        out, tau, lg = _run(dec, dev_bits(qb, c.dtype), sel, cnt, c.topk, alpha)
        assert torch.isfinite(out.float()).all()
        _check(wl, qb, sel, cnt, out, tau, lg, alpha, _scale(c))


def test_support_of_one_returns_the_value_row_exactly():
    """With a large scale the top logit leads the next by more than 1 / (alpha - 1):
    the support is that token alone, p = 1, and o is its V row, bit for bit."""
    wl = make_workload(config(2, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    sel, cnt = _selection(wl, np.random.default_rng(4), c.topk)
    qb = wl.q(0)
    scale = 40.0
    out, tau, lg = _run(dec, dev_bits(qb, c.dtype), sel, cnt, c.topk, 1.5, scale=scale)
    ob = host_bits(out)
    lg_np = lg.cpu().numpy()
    checked = 0
    for b in range(c.B):
        L = int(wl.prefill_lens[b])
        for h in range(c.H_kv):
            m = int(cnt[b, h])
            pos = O.selected_positions(sel[b, h, :m], L, c.ps)
            vs = wl.v_seq(b)[:, h, :][pos]
            for gi in range(c.G):
                z = lg_np[b, h * c.G + gi, :m * c.ps]
                z = z[np.isfinite(z)]
                top2 = np.sort(z)[-2:]
                if 0.5 * (top2[1] - top2[0]) <= 1.0 + 1e-3:
                    continue
                assert np.array_equal(ob[b, h * c.G + gi], vs[int(np.argmax(z))])
                checked += 1
    assert checked >= c.B * c.H_q // 2, checked


def test_counters_return_to_zero_and_repeat_calls_agree():
    """The split counters are back at zero after every call, and a call on the
    same inputs gives the same bits."""
    from sparse_paged_kv_page_gb300 import sa_sparse_decode_entmax, alloc_entmax_workspace
    wl = make_workload(config(5, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    sel, cnt = _selection(wl, np.random.default_rng(6), c.topk)
    q = dev_bits(wl.q(0), c.dtype)
    ws = alloc_entmax_workspace(c.B, c.H_kv, c.H_q, c.D, c.ps, c.topk)
    sel_t = torch.from_numpy(sel.astype(np.int32)).cuda()
    cnt_t = torch.from_numpy(cnt.astype(np.int32)).cuda()
    outs = []
    for _ in range(3):
        out = torch.empty((c.B, c.H_q, c.D), dtype=dec.dtype, device="cuda")
        sa_sparse_decode_entmax(dec.cache.struct, dec.batch, q, c.H_q, sel_t, cnt_t, c.topk, 1.5,
                                dec.scale, out, workspace=ws, dev_status=dec.dev_status)
        outs.append(out)
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0].view(torch.int16), o.view(torch.int16)) for o in outs[1:])
    # the counters are the workspace's last region
    from sparse_paged_kv_page_gb300 import sa_entmax_workspace_size
    n = sa_entmax_workspace_size(c.B, c.H_kv, c.H_q, c.D, c.ps, c.topk)
    tail = -(-(c.B * c.H_kv * 4) // 256) * 256
    assert int(ws[n - tail:n].to(torch.int32).sum().item()) == 0
    assert dev_status(dec) == 0


def test_empty_selection_gives_zero_and_nan():
    wl = make_workload(config(1, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    sel = np.zeros((c.B, c.H_kv, 4), dtype=np.int64)
    cnt = np.zeros((c.B, c.H_kv), dtype=np.int64)
    out, tau, _ = _run(dec, dev_bits(wl.q(0), c.dtype), sel, cnt, 4, 1.5)
    assert torch.all(out.float() == 0)
    assert torch.isnan(tau).all()
    assert dev_status(dec) == 0


def test_entmax_rejects_before_launching():
    from sparse_paged_kv_page_gb300 import SaError, sa_sparse_decode_entmax
    wl = make_workload(config(1, small=True))
    dec = make_decoder(wl)
    c = wl.cfg
    sel = torch.zeros((c.B, c.H_kv, 4), dtype=torch.int32, device="cuda")
    cnt = torch.ones((c.B, c.H_kv), dtype=torch.int32, device="cuda")
    out = torch.full((c.B, c.H_q, c.D), 7.0, dtype=dec.dtype, device="cuda")
    q = dev_bits(wl.q(0), c.dtype)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")          # zero-filled, as required
    for alpha, st in ((1.0, 1), (2.5, 1), (float("nan"), 1)):
        with pytest.raises(SaError) as e:
            sa_sparse_decode_entmax(dec.cache.struct, dec.batch, q, c.H_q, sel, cnt, 4, alpha,
                                    dec.scale, out, workspace=ws)
        assert e.value.status == st
    with pytest.raises(SaError) as e:
        sa_sparse_decode_entmax(dec.cache.struct, dec.batch, q, c.H_q, sel, cnt, 4, 1.5, dec.scale,
                                out, workspace=ws[:64])
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert torch.all(out.float() == 7.0)                     # nothing ran


@pytest.mark.parametrize("alpha", [1.5, 2.0, 1.25])
def test_many_candidates_take_the_block_solver(alpha):
    """Near-equal logits put every token within 1 of the top one: more
    candidates than one warp gathers, so the CTA-wide float64 solver runs."""
    cfg = config(3, small=True).replace(len_range=(2600, 3000), topk=170)
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    c = wl.cfg
    sel, cnt = _selection(wl, np.random.default_rng(8), c.topk)
    assert (cnt * c.ps).max() > 2048
    qb = wl.q(0)
    out, tau, lg = _run(dec, dev_bits(qb, c.dtype), sel, cnt, c.topk, alpha, scale=1e-3)
    _check(wl, qb, sel, cnt, out, tau, lg, alpha, 1e-3)
    # q = 0: every logit 0, p uniform; tau = -1/n (alpha 2), -1/sqrt(n) (alpha 1.5)
    if alpha in (1.5, 2.0):
        q0 = torch.zeros_like(dev_bits(qb, c.dtype))
        out, tau, _ = _run(dec, q0, sel, cnt, c.topk, alpha)
        t_np = tau.cpu().numpy()
        for b in range(c.B):
            L = int(wl.prefill_lens[b])
            for h in range(c.H_kv):
                n = len(O.selected_positions(sel[b, h, :cnt[b, h]], L, c.ps))
                want = -1.0 / n if alpha == 2.0 else -1.0 / np.sqrt(n)
                assert np.allclose(t_np[b, h * c.G:(h + 1) * c.G], want, rtol=1e-5, atol=0)
    assert dev_status(dec) == 0


@pytest.mark.parametrize("alpha,spread", [(1.5, 0.75), (2.0, 0.38), (1.5, 1.0)])
def test_hundreds_of_candidates_sorted_and_merged(alpha, spread):
    """Logits spread so that a few hundred entries of each row lie within
    1 / (alpha - 1) of the top one: the threshold kernel sorts per warp and
    merges; the result must still match the oracle."""
    cfg = config(3, small=True).replace(len_range=(2600, 3000), topk=170)
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    c = wl.cfg
    sel, cnt = _selection(wl, np.random.default_rng(9), c.topk)
    qb = wl.q(0)
    scale = spread * c.D ** -0.5
    out, tau, lg = _run(dec, dev_bits(qb, c.dtype), sel, cnt, c.topk, alpha, scale=scale)
    z = lg.cpu().numpy()
    m = (np.isfinite(z) & ((alpha - 1) * z > (alpha - 1) * np.nanmax(np.where(np.isfinite(z), z, -np.inf), -1, keepdims=True) - 1)).sum(-1)
    assert np.median(m) > 64 and m.max() <= 2048, (np.median(m), m.max())
    _check(wl, qb, sel, cnt, out, tau, lg, alpha, scale)
    assert dev_status(dec) == 0
