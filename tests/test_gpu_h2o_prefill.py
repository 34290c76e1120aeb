"""sa_h2o_prefill (the velox absorb / eviction with each new key as the query)
on the GPU against the oracle.

Token by token, each call is compared with the oracle's step taken from the
GPU's own state before the call (teacher forcing): retained positions equal,
scores within one bf16 ulp (the GPU's attention is float32), and where the
two choose differently the GPU's choice must be a valid one under that ulp.
One multi-token call must equal the same tokens fed one call at a time, bit
for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import dev_bits, host_bits

pytestmark = pytest.mark.gpu


def _setup(D=128, budget=24, n_sink=4, grace=6, prefill=(70, 100), structure="heavy_hitters"):
    from sparse_paged_kv_page_gb300 import PagedKVCache, make_batch
    cfg = config(4, small=True).replace(B=2, H_kv=2, H_q=8, D=D, prefill=prefill, budget=budget,
                                        n_sink=n_sink, grace=grace, decode_steps=0,
                                        structure=structure)
    wl = make_workload(cfg)
    c = wl.cfg
    cache = PagedKVCache(wl.num_blocks, c.H_kv, 1, c.D, torch.bfloat16, "cuda", with_meta=False,
                         with_hh=True)
    bt = torch.from_numpy(wl.block_table.astype(np.int32)).cuda()
    sl = torch.zeros(c.B, dtype=torch.int32, device="cuda")
    st = dict(cache=cache, bt=bt, sl=sl, batch=make_batch(bt, sl),
              ret_pos=torch.zeros((c.B, c.H_kv, budget + 1), dtype=torch.int32, device="cuda"),
              ret_cnt=torch.zeros((c.B, c.H_kv), dtype=torch.int32, device="cuda"),
              ev=torch.full((c.B, c.H_kv, 256), -1, dtype=torch.int32, device="cuda"),
              evc=torch.zeros((c.B, c.H_kv), dtype=torch.int32, device="cuda"),
              status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    return wl, st


def _append_and_absorb(wl, st, lo, hi):
    """Tokens lo .. hi-1 of every request (clipped to its prefill) in one call."""
    from sparse_paged_kv_page_gb300 import sa_append_kv, sa_h2o_prefill
    c = wl.cfg
    rows, cu = [], [0]
    for b in range(c.B):
        n = max(0, min(hi, int(wl.prefill_lens[b])) - lo)
        if n:
            rows.append(wl.k_pre[wl.pre_cu[b] + lo:wl.pre_cu[b] + lo + n])
        cu.append(cu[-1] + n)
    if cu[-1] == 0:
        return False
    k = dev_bits(np.concatenate(rows), "bf16")
    new_cu = torch.tensor(cu, dtype=torch.int32, device="cuda")
    mx = max(cu[i + 1] - cu[i] for i in range(c.B))
    sa_append_kv(st["cache"].struct, st["batch"], k, k, new_cu, mx, hh=st["cache"].hh,
                 dev_status=st["status"])
    sa_h2o_prefill(st["cache"].struct, st["batch"], new_cu, st["cache"].hh,
                   st["cache"].hh.shape[0], st["ret_pos"], st["ret_cnt"], c.budget + 1, c.budget,
                   c.n_sink, c.grace, c.decay, c.scale, evicted=st["ev"], evicted_cnt=st["evc"],
                   dev_status=st["status"])
    return True


def _gpu_state(wl, st, b, h):
    cnt = int(st["ret_cnt"][b, h])
    pos = st["ret_pos"][b, h, :cnt].cpu().numpy().astype(np.int64)
    hh = O.decode_kdt(host_bits(st["cache"].hh)[wl.block_table[b, pos], h], "bf16")
    return pos, hh


@pytest.mark.parametrize("D", [128, 64])
def test_token_by_token_against_oracle(D):
    wl, st = _setup(D=D)
    c = wl.cfg
    kf = {(b, h): O.decode_kdt(wl.k_pre[wl.pre_cu[b]:wl.pre_cu[b + 1], h], "bf16")
          for b in range(c.B) for h in range(c.H_kv)}
    agree = total = 0
    for t in range(int(wl.prefill_lens.max())):
        before = {(b, h): _gpu_state(wl, st, b, h) for b in range(c.B) for h in range(c.H_kv)}
        assert _append_and_absorb(wl, st, t, t + 1)
        torch.cuda.synchronize()
        evc = st["evc"].cpu().numpy()
        ev = st["ev"].cpu().numpy()
        for b in range(c.B):
            if t >= int(wl.prefill_lens[b]):
                continue
            for h in range(c.H_kv):
                pos0, hh0 = before[(b, h)]
                keys0 = kf[(b, h)][pos0]
                _, pos_o, hh_o, ev_o = O.h2o_proxy_token(
                    keys0, pos0, hh0, kf[(b, h)][t], t, decay=c.decay, budget=c.budget,
                    n_sink=c.n_sink, grace=c.grace, scale=c.scale)
                pos_g, hh_g = _gpu_state(wl, st, b, h)
                total += 1
                assert len(pos_g) == min(t + 1, c.budget)
                assert pos_g[:c.n_sink].tolist() == list(range(min(c.n_sink, t + 1)))
                assert pos_g[-c.grace:].tolist() == list(range(max(0, t + 1 - c.grace), t + 1))
                if np.array_equal(pos_g, pos_o):
                    agree += 1
                    ulp = O.ulp_kdt(np.maximum(hh_g, hh_o), "bf16")
                    assert np.all(np.abs(hh_g - hh_o) <= ulp), (t, b, h)
                    if ev_o is not None:
                        assert int(evc[b, h]) == 1 and int(ev[b, h, 0]) == ev_o
                else:
                    # a near tie decided the other way: the GPU's pick must be a
                    # minimum of the oracle's folded scores within one ulp
                    assert ev_o is not None and int(evc[b, h]) == 1
                    full_pos = np.append(pos0, t)
                    full_hh = np.append(O.h2o_store(c.decay * hh0 + _attn(keys0, kf[(b, h)][t], c.scale)), 0.0)
                    gi = int(np.nonzero(full_pos == ev[b, h, 0])[0][0])
                    elig = np.arange(c.n_sink, len(full_pos) - c.grace)
                    assert gi in elig
                    tol = O.ulp_kdt(full_hh, "bf16")
                    assert full_hh[gi] - tol[gi] <= (full_hh[elig] + tol[elig]).min()
    assert int(st["status"].item()) == 0
    assert agree >= 0.95 * total, (agree, total)


def _attn(keys, k, scale):
    z = keys @ k * scale
    p = np.exp(z - z.max())
    return p / p.sum()


def test_one_call_equals_token_by_token():
    wl, a = _setup()
    _, b = _setup()
    c = wl.cfg
    assert _append_and_absorb(wl, a, 0, 1000)                 # every token in one call
    t = 0
    while _append_and_absorb(wl, b, t, t + 1):
        t += 1
    torch.cuda.synchronize()
    assert torch.equal(a["ret_cnt"], b["ret_cnt"])
    for r in range(c.B):
        for h in range(c.H_kv):
            n = int(a["ret_cnt"][r, h])
            assert torch.equal(a["ret_pos"][r, h, :n], b["ret_pos"][r, h, :n])
            # the retained entries' scores (an evicted slot keeps whatever it last held)
            pa, ha = _gpu_state(wl, a, r, h)
            pb, hb = _gpu_state(wl, b, r, h)
            assert np.array_equal(ha, hb)
    assert int(a["status"].item()) == 0 and int(b["status"].item()) == 0


def test_below_budget_keeps_everything_and_matches_the_oracle():
    wl, st = _setup(budget=200, prefill=(60, 90))
    c = wl.cfg
    assert _append_and_absorb(wl, st, 0, 1000)
    torch.cuda.synchronize()
    for b in range(c.B):
        for h in range(c.H_kv):
            L = int(wl.prefill_lens[b])
            pos_g, hh_g = _gpu_state(wl, st, b, h)
            assert pos_g.tolist() == list(range(L))
            keys = O.decode_kdt(wl.k_pre[wl.pre_cu[b]:wl.pre_cu[b + 1], h], "bf16")
            _, pos_o, hh_o, ev = O.h2o_proxy_prefill(keys, np.arange(L), decay=c.decay, budget=c.budget,
                                                     n_sink=c.n_sink, grace=c.grace, scale=c.scale)
            assert ev == [] and pos_o.tolist() == pos_g.tolist()
            # scores rounded to bf16 at every fold: allow a few ulps of drift over the prefill
            assert np.all(np.abs(hh_g - hh_o) <= 4 * O.ulp_kdt(np.maximum(hh_g, hh_o), "bf16") + 1e-6)


def test_decoder_with_trimmed_prefill_then_decode_steps():
    """A token-level decoder whose prefill goes through the absorb / eviction
    holds `budget` entries after the prefill, with the oracle's retained set,
    and then decodes with the decode-side update as usual."""
    from gpu_util import make_decoder, step_inputs
    cfg = config(4, small=True).replace(B=2, H_kv=2, H_q=8, prefill=(150, 200), budget=48,
                                        n_sink=4, grace=8, decode_steps=4, structure="heavy_hitters")
    wl = make_workload(cfg)
    c = wl.cfg
    dec = make_decoder(wl, extra=dict(proxy_prefill=True))
    rc = dec.ret_cnt.cpu().numpy()
    assert np.all(rc == c.budget)
    agree = 0
    for b in range(c.B):
        for h in range(c.H_kv):
            L = int(wl.prefill_lens[b])
            keys = O.decode_kdt(wl.k_pre[wl.pre_cu[b]:wl.pre_cu[b + 1], h], "bf16")
            _, pos_o, _, _ = O.h2o_proxy_prefill(keys, np.arange(L), decay=c.decay, budget=c.budget,
                                                 n_sink=c.n_sink, grace=c.grace, scale=c.scale)
            got = dec.ret_pos[b, h, :c.budget].cpu().numpy()
            agree += int(np.array_equal(got, pos_o))
            assert got[:c.n_sink].tolist() == list(range(c.n_sink))
            assert got[-c.grace:].tolist() == list(range(L - c.grace, L))
    assert agree >= c.B * c.H_kv - 1, agree          # an ulp-level tie may decide one unit the other way
    for t in range(c.decode_steps):
        dec.step(*step_inputs(wl, t))
    torch.cuda.synchronize()
    assert np.all(dec.ret_cnt.cpu().numpy() == c.budget)
    assert int(dec.dev_status.item()) == 0
