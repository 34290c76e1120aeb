"""sa_h2o_update (and the token-level step) on the GPU against the oracle.

* fold: bf16 hh within 1 ulp of the oracle's once-rounded float64 fold;
* eviction: bit-exact wherever the GPU's and the oracle's bf16 scores agree,
  and otherwise a valid choice under the scores' tolerance; sink / grace /
  budget invariants always; along whole trajectories, teacher forced, the
  oracle's eviction of the GPU's own folded scores equals the GPU's, bit for bit;
* exact case: zero probabilities make the fold exact on both sides, so the
  evictions (heavy ties included) must match bit for bit;
* the vortex page's oracle checks on a long run without eviction: probability
  mass near the 1/(1-decay) steady state, small relative error against a
  float64 accumulator, top-k agreement where the boundary is wider than 1 ulp.
"""
import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden
from sa_synth import config, make_workload
from gpu_util import make_decoder, step_inputs, dev_status, host_bits, h2o_teacher_forced

pytestmark = pytest.mark.gpu


def _run_update(hh_bits, logits, lse, ret, cnt, bt, G, budget, n_sink, grace, decay, window=False):
    from sparse_paged_kv_page_gb300 import make_batch, sa_h2o_update, sa_h2o_update_window
    B, H, cap = ret.shape
    nslots = hh_bits.shape[0]
    hh = torch.from_numpy(hh_bits.view(np.int16)).cuda().view(torch.bfloat16)
    lg = torch.from_numpy(logits.astype(np.float32)).cuda()
    ls = torch.from_numpy(lse.astype(np.float32)).cuda()
    rp = torch.from_numpy(ret.astype(np.int32)).cuda()
    rc = torch.from_numpy(cnt.astype(np.int32)).cuda()
    btt = torch.from_numpy(bt.astype(np.int32)).cuda()
    sl = torch.full((B,), bt.shape[1], dtype=torch.int32, device="cuda")
    ev = torch.full((B, H, cap), -1, dtype=torch.int32, device="cuda")
    evc = torch.zeros((B, H), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = sa_h2o_update_window if window else sa_h2o_update
    fn(make_batch(btt, sl), H, H * G, lg, cap, ls, hh, nslots, rp, rc, cap, budget,
       n_sink, grace, decay, evicted=ev, evicted_cnt=evc, dev_status=st)
    torch.cuda.synchronize()
    return (host_bits(hh), rp.cpu().numpy(), rc.cpu().numpy(), ev.cpu().numpy(),
            evc.cpu().numpy(), int(st.item()))


def _inputs(rng, B, H, G, n, cap, L, zero_probs=False, tie_vals=None):
    nslots = B * L + 7
    bt = rng.permutation(nslots)[:B * L].reshape(B, L).astype(np.int32)   # disjoint slots
    ret = np.zeros((B, H, cap), dtype=np.int64)
    cnt = np.full((B, H), n, dtype=np.int64)
    for b in range(B):
        for h in range(H):
            ret[b, h, :n] = np.sort(rng.choice(L, size=n, replace=False))
    if tie_vals is not None:
        vals = rng.choice(np.asarray(tie_vals), size=nslots * H)
    else:
        vals = np.abs(rng.standard_normal(nslots * H)) * rng.choice([0.01, 0.1, 1.0], size=nslots * H)
    hh_bits = O.encode_kdt(vals, "bf16").reshape(nslots, H)
    z = rng.standard_normal((B, H * G, cap)) * 2.0
    if zero_probs:
        z[:] = -np.inf
    lse = rng.standard_normal((B, H * G)) + 5.0
    return hh_bits, z, lse, ret, cnt, bt


def _oracle(hh_bits, z, lse, ret, cnt, bt, G, budget, n_sink, grace, decay, window=False):
    B, H, _ = ret.shape
    res = {}
    for b in range(B):
        for h in range(H):
            n = int(cnt[b, h])
            pos = ret[b, h, :n]
            slots = bt[b, pos]
            hh = O.decode_kdt(hh_bits[slots, h], "bf16")
            zz = z[b, h * G:(h + 1) * G, :n]
            ex = (O.h2o_fold_window(hh, zz, n_sink, grace, decay) if window
                  else O.h2o_fold(hh, zz, lse[b, h * G:(h + 1) * G], decay))
            hb = O.h2o_store(ex)
            kept, _, evd = O.h2o_evict(hb, pos, budget, n_sink, grace)
            res[(b, h)] = (slots, hb, kept, sorted(evd))
    return res


def _check_eviction_valid(kept, pos, vals, budget, n_sink, grace, tol):
    n = len(pos)
    assert len(kept) == min(n, budget)
    assert np.all(np.diff(kept) > 0) and set(kept) <= set(pos.tolist())
    assert kept[:n_sink].tolist() == pos[:n_sink].tolist()
    if grace:
        assert kept[-grace:].tolist() == pos[-grace:].tolist()
    gone = np.isin(pos, kept, invert=True)
    elig = np.zeros(n, dtype=bool)
    elig[n_sink:n - grace] = True
    if gone.any() and (elig & ~gone).any():
        assert (vals - tol)[gone].max() <= (vals + tol)[elig & ~gone].min()


@pytest.mark.parametrize("window", [False, True])
@pytest.mark.parametrize("n,budget", [(700, 512), (513, 512), (100, 512), (4097, 512)])
def test_fold_and_evict_generated_inputs(n, budget, window):
    rng = np.random.default_rng([n, budget])
    B, H, G, cap, L = 2, 3, 4, 4200, 5000
    n_sink, grace, decay = 4, 16, 0.984375
    args = _inputs(rng, B, H, G, n, cap, L)
    hh_bits, z, lse, ret, cnt, bt = args
    got_hh, rp, rc, ev, evc, st = _run_update(*args, G, budget, n_sink, grace, decay, window)
    assert st == 0
    want = _oracle(*args, G, budget, n_sink, grace, decay, window)
    for (b, h), (slots, hb, kept, evd) in want.items():
        g = O.decode_kdt(got_hh[slots, h], "bf16")
        ulp = O.ulp_kdt(np.maximum(np.abs(g), np.abs(hb)), "bf16")
        assert np.all(np.abs(g - hb) <= ulp), (b, h)
        k = int(rc[b, h])
        gk = rp[b, h, :k]
        pos = ret[b, h, :int(cnt[b, h])]
        assert int(evc[b, h]) == len(pos) - k
        assert np.array_equal(np.sort(np.concatenate([gk, ev[b, h, :evc[b, h]]])), pos)
        if np.array_equal(g, hb):
            assert np.array_equal(gk, kept) and ev[b, h, :evc[b, h]].tolist() == evd
        else:
            _check_eviction_valid(gk, pos, hb, budget, n_sink, grace, O.ulp_kdt(hb, "bf16"))


@pytest.mark.parametrize("ties", [[0.0, 0.5, 1.0], [0.25], [0.0, 1e-3, 2e-3, 3e-3]])
@pytest.mark.parametrize("n_sink,grace", [(4, 16), (0, 0), (0, 5), (3, 0)])
def test_exact_eviction_when_probabilities_vanish(ties, n_sink, grace):
    rng = np.random.default_rng([len(ties), n_sink, grace])
    B, H, G, cap, L, n, budget = 2, 2, 4, 1200, 1500, 1000, 300
    args = _inputs(rng, B, H, G, n, cap, L, zero_probs=True, tie_vals=ties)
    got_hh, rp, rc, ev, evc, st = _run_update(*args, G, budget, n_sink, grace, 0.984375)
    want = _oracle(*args, G, budget, n_sink, grace, 0.984375)
    for (b, h), (slots, hb, kept, evd) in want.items():
        assert np.array_equal(O.decode_kdt(got_hh[slots, h], "bf16"), hb)
        assert np.array_equal(rp[b, h, :rc[b, h]], kept)
        assert ev[b, h, :evc[b, h]].tolist() == evd


def _oracle_traj_init(wl):
    c = wl.cfg
    st = {}
    for b in range(c.B):
        for h in range(c.H_kv):
            L = int(wl.prefill_lens[b])
            st[(b, h)] = {"pos": np.arange(L), "hh": np.zeros(L), "ex": np.zeros(L)}
    return st


def _oracle_traj_step(wl, st, t, qb, window=False):
    c = wl.cfg
    for (b, h), s in st.items():
        L = wl.seq_len(b, t + 1)
        s["pos"] = np.append(s["pos"], L - 1)
        s["hh"] = np.append(s["hh"], 0.0)
        s["ex"] = np.append(s["ex"], 0.0)
        ks = wl.k_seq(b, t + 1)[:, h, :]
        vs = wl.v_seq(b, t + 1)[:, h, :]
        r = O.h2o_unit_step(s["hh"], s["pos"], ks, vs, qb[b, h * c.G:(h + 1) * c.G],
                            dtype=c.dtype, decay=c.decay, budget=c.budget, n_sink=c.n_sink,
                            grace=c.grace, scale=c.scale, window_softmax=window)
        s["ex"] = (O.h2o_fold_window(s["ex"], r["logits"], c.n_sink, c.grace, c.decay) if window
                   else O.h2o_fold(s["ex"], r["logits"], r["lse"], c.decay))
        s["last"] = r
        keep = np.isin(s["pos"], r["kept"])
        s["pos"], s["hh"], s["ex"] = s["pos"][keep], r["hh_bf16"][keep], s["ex"][keep]


@pytest.mark.parametrize("window", [False, True])
def test_token_level_trajectory_small(window):
    """Every unit of the reduced token-level workload, at every step, teacher
    forced: the oracle starts from the GPU's retained list and bf16 scores;
    folded scores within 1 ulp, evictions bit-exact on the GPU's scores."""
    wl = make_workload(config(4, small=True))
    c = wl.cfg
    dec = make_decoder(wl, extra=dict(window_softmax=window))
    units = [(b, h) for b in range(c.B) for h in range(c.H_kv)]
    assert h2o_teacher_forced(dec, wl, units, c.decode_steps, window=window) == len(units) * c.decode_steps
    assert dev_status(dec) == 0


def test_vortex_mass_and_accuracy_without_eviction():
    g = golden("vortex_h2o_constants.txt")
    decay = float(g["default_decay"])
    T = 300
    cfg = config(4, small=True).replace(B=2, H_q=8, H_kv=2, prefill=(128, 128), decode_steps=T,
                                        budget=10 ** 6, structure="heavy_hitters")
    wl = make_workload(cfg)
    dec = make_decoder(wl)
    ost = _oracle_traj_init(wl)
    for t in range(T):
        q, kn, vn = step_inputs(wl, t)
        dec.step(q, kn, vn)
        _oracle_traj_step(wl, ost, t, wl.q(t))
    torch.cuda.synchronize()
    hh = host_bits(dec.cache.hh)
    closed = (1 - decay ** T) / (1 - decay)
    for (b, h), s in ost.items():
        got = O.decode_kdt(hh[wl.block_table[b, s["pos"]], h], "bf16")
        assert abs(s["ex"].sum() - closed) < 1e-9 * closed           # float64 recurrence
        lost = 1.0 - got.sum() / closed
        assert lost < float(g["oracle_mass_lost_fail"]), lost
        rel = np.abs(got - s["ex"]).max() / np.abs(s["ex"]).max()
        assert rel < float(g["recurrence_rel_err_max"]), rel
        # top-k: the GPU's bf16 accumulator against the oracle's own bf16 one
        # (same recurrence, same storage rounding) wherever the oracle's
        # boundary is wider than the 16-ulp GPU/oracle bound of the trajectory.
        k = int(g["recurrence_topk"])
        ob = s["hh"]
        srt = np.sort(ob)[::-1]
        gap, ulp = srt[k - 1] - srt[k], float(O.ulp_kdt(srt[k - 1], "bf16"))
        if gap > 16 * ulp:
            assert set(np.argsort(-got, kind="stable")[:k]) == set(np.argsort(-ob, kind="stable")[:k])
    assert dev_status(dec) == 0
