"""Helpers for the GPU parity tests: move generator inputs to the device, build
a decoder for a workload, and the comparison rules used throughout.

Inputs always come from sa_synth; expected values always come from oracle/.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from sa_synth import Workload, fill_stale

TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def dev_bits(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """uint16 bit patterns -> a CUDA tensor of the bf16/fp16 dtype (bit-exact)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TDT[dtype])


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_decoder(wl: Workload, stale: str = "normal3", extra=None):
    """A SparseDecoder for the workload, pools filled with stale contents, prefilled."""
    from sparse_paged_kv_page_gb300.step import SparseDecoder
    c = wl.cfg
    token = c.ps == 1 and c.budget > 0
    kw = dict(batch=c.B, num_q_heads=c.H_q, num_kv_heads=c.H_kv, head_dim=c.D, page_size=c.ps,
              num_blocks=wl.num_blocks, bt_stride=wl.max_pages, dtype=TDT[c.dtype],
              scale=c.scale)
    if token:
        cap = int(wl.prefill_lens.max()) + wl.total_steps + 1
        kw.update(budget=c.budget, n_sink=c.n_sink, grace=c.grace, decay=c.decay, ret_cap=cap)
    else:
        kw.update(topk=c.topk, w_avg=c.w_avg, w_peak=c.w_peak)
    if extra:
        kw.update(extra)
    dec = SparseDecoder(**kw)
    fill_stale(dec.cache.k, stale, 11)
    fill_stale(dec.cache.v, stale, 12)
    if dec.cache.meta is not None:
        fill_stale(dec.cache.meta, stale, 13)
    if dec.cache.hh is not None:
        dec.cache.hh.fill_(7.5)                       # stale scores of recycled slots
    dec.set_block_table(torch.from_numpy(wl.block_table))
    dec.prefill(dev_bits(wl.k_pre, c.dtype), dev_bits(wl.v_pre, c.dtype), wl.prefill_lens.tolist())
    torch.cuda.synchronize()
    return dec


def step_inputs(wl: Workload, t: int, device="cuda"):
    c = wl.cfg
    q = dev_bits(wl.q(t), c.dtype, device)
    kn, vn = wl.kv_new(t)
    return q, dev_bits(kn, c.dtype, device), dev_bits(vn, c.dtype, device)


def dev_status(dec) -> int:
    return int(dec.dev_status.item())


# ---------------------------------------------------------------------------
# comparison rules
# ---------------------------------------------------------------------------
def score_norm(mn, mx, me, q, w_avg, w_peak):
    """Norm-wise scale of a page score: (1/G) sum_g sum_d (w_avg |q mean| + w_peak |q| max(|M|,|m|))."""
    aq = np.abs(q)
    big = np.maximum(np.abs(mx), np.abs(mn))
    return (abs(w_avg) * (np.abs(me) @ aq.T) + abs(w_peak) * (big @ aq.T)).mean(1)


def assert_scores(got, want, norm, rel=1e-4):
    err = np.abs(got.astype(np.float64) - want)
    bound = rel * np.maximum(np.abs(want), norm)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, f"{bad.size} scores off: first p={bad[:5]}, err={err[bad[:5]]}, bound={bound[bad[:5]]}"


def score_error_bound(norm, D, G):
    """Worst-case float32 error of the linearised score: (3D + G + 4) u A."""
    return (3 * D + G + 4) * 2.0 ** -24 * norm


def assert_selection_valid(sel, S, eps, n, topk):
    """The GPU's selection is a correct top-k for some scores within eps of the
    oracle's: tail kept, ascending, right count, and no unselected candidate can
    outrank a selected one."""
    sel = list(sel)
    if n <= topk:
        assert sel == list(range(n)), sel
        return True
    assert len(sel) == topk and sel[-1] == n - 1 and sel == sorted(set(sel)), sel
    X = np.array(sel[:-1])
    mask = np.zeros(n - 1, dtype=bool)
    mask[X] = True
    if mask.all() or not mask.any():
        return True
    lo = (S[:n - 1] + eps[:n - 1])[mask].min()
    hi = (S[:n - 1] - eps[:n - 1])[~mask].max()
    assert lo >= hi, f"selection not valid: weakest kept {lo} < strongest dropped {hi}"
    return True


def assert_attention(got_o, want_o, got_lse=None, want_lse=None, atol=2e-2, rtol=2e-2, lse_tol=1e-3):
    got_o = np.asarray(got_o, dtype=np.float64)
    err = np.abs(got_o - want_o)
    bad = err > atol + rtol * np.abs(want_o)
    assert not bad.any(), f"{bad.sum()} outputs off, max err {err.max()}"
    if want_lse is not None:
        gl = np.asarray(got_lse, dtype=np.float64)
        fin = np.isfinite(want_lse)
        assert np.array_equal(np.isfinite(gl), fin), (gl, want_lse)
        assert np.all(gl[~fin] == -np.inf)
        if fin.any():
            assert np.abs(gl[fin] - want_lse[fin]).max() < lse_tol


def oracle_unit(wl: Workload, b: int, h: int, steps_done: int, q_bits):
    """Oracle of one (request, KV head) after `steps_done` appends, for query q_bits [H_q, D]."""
    c = wl.cfg
    L = wl.seq_len(b, steps_done)
    ks = wl.k_seq(b, steps_done, head=h)
    vs = wl.v_seq(b, steps_done, head=h)
    qg = q_bits[h * c.G:(h + 1) * c.G]
    return O.page_decode_unit(ks, vs, L, qg, ps=c.ps, topk=c.topk, w_avg=c.w_avg,
                              w_peak=c.w_peak, dtype=c.dtype, scale=c.scale), ks, vs, qg, L


def h2o_teacher_forced(dec, wl, units, steps, window=False, every_unit_invariants=True):
    """Run `steps` token-level decode steps on the GPU and check each sampled
    (request, KV head) unit at every step against the oracle started from the
    GPU's own state before that step: its retained list and its bf16 scores.

    Per unit and step:
      * attention output of the step within atol 2e-2 + rtol 2e-2;
      * the GPU's folded bf16 score of every entry (the new token included)
        within 1 bf16 ulp of the oracle's once-rounded float64 fold;
      * the oracle's eviction rule applied to the GPU's own folded bf16
        scores reproduces the GPU's retained list and its evicted positions
        bit for bit (the rule is exact integer / bf16 comparison, so this is
        the form in which eviction parity is well defined).
    Every unit (sampled or not) keeps the budget, sinks and grace entries.
    Returns the number of (unit, step) checks made."""
    c = wl.cfg
    bt = wl.block_table
    rows = lambda h: slice(h * c.G, (h + 1) * c.G)
    rp, rc = dec.ret_pos.cpu().numpy(), dec.ret_cnt.cpu().numpy()
    hh = host_bits(dec.cache.hh)
    prev = {}
    for b, h in units:
        pos = rp[b, h, :rc[b, h]].astype(np.int64)
        prev[(b, h)] = (pos, O.decode_kdt(hh[bt[b, pos], h], "bf16"))
    checks = 0
    for t in range(steps):
        q, kn, vn = step_inputs(wl, t)
        dec.step(q, kn, vn)
        torch.cuda.synchronize()
        rp, rc = dec.ret_pos.cpu().numpy(), dec.ret_cnt.cpu().numpy()
        ev, evc = dec.evicted.cpu().numpy(), dec.evicted_cnt.cpu().numpy()
        hh = host_bits(dec.cache.hh)
        out = dec.out.float().cpu().numpy()
        qb = wl.q(t)
        if every_unit_invariants:
            for b in range(c.B):
                L = wl.seq_len(b, t + 1)
                for h in range(c.H_kv):
                    k = int(rc[b, h])
                    assert k == min(c.budget, L), (t, b, h, k)
                    gk = rp[b, h, :k]
                    assert gk[:c.n_sink].tolist() == list(range(c.n_sink))
                    if c.grace:
                        assert gk[-c.grace:].tolist() == list(range(L - c.grace, L))
        for b, h in units:
            pos0, hb0 = prev[(b, h)]
            L = wl.seq_len(b, t + 1)
            assert L - 1 not in set(pos0.tolist())
            pos = np.append(pos0, L - 1)
            hb = np.append(hb0, 0.0)                  # zeroed on write by the append
            r = O.h2o_unit_step(hb, pos, wl.k_seq(b, t + 1, head=h), wl.v_seq(b, t + 1, head=h),
                                qb[b, rows(h)], dtype=c.dtype, decay=c.decay, budget=c.budget,
                                n_sink=c.n_sink, grace=c.grace, scale=c.scale,
                                window_softmax=window)
            assert_attention(out[b, rows(h)], r["out"])
            g = O.decode_kdt(hh[bt[b, pos], h], "bf16")      # the GPU's folded score of every entry
            ulp = O.ulp_kdt(np.maximum(np.abs(g), np.abs(r["hh_bf16"])), "bf16")
            bad = np.abs(g - r["hh_bf16"]) > ulp
            assert not bad.any(), (t, b, h, np.nonzero(bad)[0][:5])
            kept, _, evd = O.h2o_evict(g, pos, c.budget, c.n_sink, c.grace)
            gk = rp[b, h, :rc[b, h]].astype(np.int64)
            assert np.array_equal(gk, kept), (t, b, h)
            assert ev[b, h, :evc[b, h]].tolist() == sorted(evd), (t, b, h)
            prev[(b, h)] = (gk, g[np.isin(pos, gk)])
            checks += 1
    return checks
