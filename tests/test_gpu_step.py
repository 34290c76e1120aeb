"""sa_decode_step (append, score, select and decode chained by programmatic
dependent launch) against the same step made of the four separate calls, on
twin decoders built from the same seeded workload: every output and every
piece of cache state must be bit-identical, except the score entry of the
page a one-token append wrote (the step scores it beside the append; it is
always selected). The separate calls themselves are checked against the
oracle in the other GPU test files.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import make_decoder, dev_bits, dev_status, host_bits, step_inputs

pytestmark = pytest.mark.gpu


def _twins(cid, small=True):
    wl = make_workload(config(cid, small=small))
    return wl, make_decoder(wl), make_decoder(wl)


def _state(dec):
    return dict(k=host_bits(dec.cache.k), v=host_bits(dec.cache.v), meta=host_bits(dec.cache.meta),
                seq=dec.seq_lens.cpu().numpy(), sel=dec.sel_idx.cpu().numpy(),
                cnt=dec.sel_cnt.cpu().numpy(), out=host_bits(dec.out),
                lse=dec.lse.cpu().numpy().view(np.uint32), scores=dec.scores.cpu().numpy())


def _compare(a, b, wl, tail_unspecified):
    for key in ("k", "v", "meta", "seq", "sel", "cnt", "out", "lse"):
        assert np.array_equal(a[key], b[key]), key
    c = wl.cfg
    for bi in range(c.B):
        n = O.num_pages(int(a["seq"][bi]), c.ps)
        m = n - 1 if tail_unspecified else n
        sa, sb = a["scores"][bi, :, :m], b["scores"][bi, :, :m]
        assert np.array_equal(sa.view(np.uint32), sb.view(np.uint32)), bi


@pytest.mark.parametrize("cid,small", [(2, True), (5, True), (2, False)])
def test_step_matches_separate_calls_with_append(cid, small):
    wl, fused, split = _twins(cid, small)
    steps = min(wl.total_steps, 24)
    for t in range(steps):
        q, kn, vn = step_inputs(wl, t)
        fused.step(q, kn, vn)
        split.append(kn, vn)
        split.attend(q)
        torch.cuda.synchronize()
        _compare(_state(fused), _state(split), wl, tail_unspecified=True)
    assert dev_status(fused) == 0 and dev_status(split) == 0
    assert fused.seq_lens.cpu().tolist() == [wl.seq_len(b, steps) for b in range(wl.cfg.B)]


def test_step_with_reserved_pages_matches_separate_calls():
    wl = make_workload(config(2, small=False))
    extra = dict(n_bos=2, n_eos=3)
    fused, split = make_decoder(wl, extra=extra), make_decoder(wl, extra=extra)
    for t in range(6):
        q, kn, vn = step_inputs(wl, t)
        fused.step(q, kn, vn)
        split.append(kn, vn)
        split.attend(q)
        torch.cuda.synchronize()
        _compare(_state(fused), _state(split), wl, tail_unspecified=True)
        cnt = fused.sel_cnt.cpu().numpy()
        sel = fused.sel_idx.cpu().numpy()
        for b in range(wl.cfg.B):
            n = O.num_pages(wl.seq_len(b, t + 1), wl.cfg.ps)
            for h in range(wl.cfg.H_kv):
                s = sel[b, h, :cnt[b, h]]
                assert s[:2].tolist() == [0, 1] and s[-3:].tolist() == [n - 3, n - 2, n - 1]
    assert dev_status(fused) == 0


@pytest.mark.parametrize("cid", [1, 3])
def test_step_without_append_is_exact(cid):
    wl, fused, split = _twins(cid)
    q = dev_bits(wl.q(0), wl.cfg.dtype)
    fused.step(q)
    split.attend(q)
    torch.cuda.synchronize()
    _compare(_state(fused), _state(split), wl, tail_unspecified=False)


def test_step_multi_token_append_runs_first():
    """More than one new token per request: the append precedes the scorer and
    every score is exact, including pages that stopped being the tail."""
    from sparse_paged_kv_page_gb300 import sa_append_kv, sa_decode_step
    wl = make_workload(config(3, small=True))
    c = wl.cfg
    # three spare blocks per request past the prefill's pages, so appends cross pages
    extra = dict(num_blocks=wl.num_blocks + 3 * c.B)
    fused, split = make_decoder(wl, extra=extra), make_decoder(wl, extra=extra)
    bt = wl.block_table.copy()
    nxt = wl.num_blocks
    for b in range(c.B):
        free = np.nonzero(bt[b] < 0)[0][:3]
        bt[b, free] = nxt + np.arange(len(free))
        nxt += len(free)
    for d in (fused, split):
        d.set_block_table(torch.from_numpy(bt))
    rng = np.random.default_rng(5)
    room = (bt >= 0).sum(1) * c.ps - wl.prefill_lens   # what the block table holds
    n_new = np.minimum(rng.integers(0, 2 * c.ps + 3, size=c.B), room)
    assert np.any((wl.prefill_lens % c.ps) + n_new > c.ps)   # some old tail stops being the tail
    cu = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    T = int(cu[-1])
    k = dev_bits(rng.integers(0, 1 << 16, size=(T, c.H_kv, c.D)).astype(np.uint16) & 0xBFFF, c.dtype)
    v = dev_bits(rng.integers(0, 1 << 16, size=(T, c.H_kv, c.D)).astype(np.uint16) & 0xBFFF, c.dtype)
    new_cu = torch.from_numpy(cu).cuda()
    q = dev_bits(wl.q(0), c.dtype)
    mx = int(n_new.max())
    sa_decode_step(fused.cache.struct, fused.batch, k, v, new_cu, mx, q, c.H_q, c.w_avg, c.w_peak,
                   fused.scores, fused.max_pages, c.topk, fused.sel_idx, fused.sel_cnt, fused.scale,
                   fused.out, lse=fused.lse, workspace=fused.workspace, dev_status=fused.dev_status)
    sa_append_kv(split.cache.struct, split.batch, k, v, new_cu, mx, dev_status=split.dev_status)
    split.attend(q)
    torch.cuda.synchronize()
    _compare(_state(fused), _state(split), wl, tail_unspecified=False)
    assert fused.seq_lens.cpu().tolist() == [int(wl.prefill_lens[b] + n_new[b]) for b in range(c.B)]
    assert dev_status(fused) == 0 and dev_status(split) == 0


def test_step_rejects_before_launching():
    from sparse_paged_kv_page_gb300 import SaError, sa_decode_step
    wl, dec, _ = _twins(2)
    c = wl.cfg
    q, kn, vn = step_inputs(wl, 0)
    seq0 = dec.seq_lens.clone()
    args = (dec.cache.struct, dec.batch, kn, vn, dec.decode_cu, 1, q, c.H_q, c.w_avg, c.w_peak,
            dec.scores, dec.max_pages, c.topk, dec.sel_idx, dec.sel_cnt, dec.scale, dec.out)
    with pytest.raises(SaError) as e:
        sa_decode_step(*args, lse=dec.lse, workspace=None, dev_status=dec.dev_status)
    assert e.value.status == 3
    with pytest.raises(SaError) as e:
        sa_decode_step(*args[:3], None, *args[4:], lse=dec.lse, workspace=dec.workspace)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert torch.equal(dec.seq_lens, seq0)            # nothing ran
