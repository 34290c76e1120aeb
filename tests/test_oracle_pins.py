"""Pins of the CPU oracle to things other than itself.

Each group ties one oracle function to a library routine, a brute-force
enumeration, a closed form, an invariant the pages state, or a value the
pages print (fixtures under tests/golden). Chosen so that a plausible slip
(a dropped envelope, a wrong sign, a missing 1/f, a transposed operand, a
wrong tie-break, double rounding) fails at least one of them.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def _bf16_bits_torch(x32):
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_decode_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=20000, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = O.decode_kdt(bits, "bf16")
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])
    ref16 = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    got16 = O.decode_kdt(bits, "fp16")
    m = ~np.isnan(ref16)
    assert np.array_equal(ref16[m], got16[m])


def test_round_bf16_matches_torch_float32_cast():
    # float32 inputs are exact in float64, so one rounding from float64 equals
    # torch's single rounding from float32 (round to nearest even).
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(50000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),     # subnormal range
        (rng.standard_normal(5000) * 3e38).astype(np.float32),      # near overflow
        np.array([0.0, -0.0, np.inf, -np.inf], dtype=np.float32),
    ])
    # exact ties: a bf16 value plus half its spacing
    base = _bf16_bits_torch(rng.standard_normal(5000).astype(np.float32))
    b64 = O.decode_kdt(base, "bf16")
    ties = (b64 + 0.5 * O.ulp_kdt(b64, "bf16")).astype(np.float32)
    x = np.concatenate([x, ties])
    assert np.array_equal(O.encode_kdt(x.astype(np.float64), "bf16"), _bf16_bits_torch(x))


def test_round_fp16_matches_numpy_direct_cast():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(50000) * s for s in (1.0, 1e-6, 3e4, 1e5)])
    x = np.concatenate([x, [0.0, -0.0, 65504.0, 65520.0, 65519.99, 2.0 ** -25, 2.0 ** -24]])
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.encode_kdt(x, "fp16"), ref)


def test_round_once_not_twice():
    # A float64 value just above a bf16 midpoint must round up; rounding to
    # float32 first would land exactly on the midpoint and round to even (down).
    one = 1.0
    mid = one + 2.0 ** -8                 # midpoint between 1 and 1 + 2^-7
    x = mid + 2.0 ** -40                  # above it, but collapses onto it in float32
    assert float(np.float32(x)) == mid
    assert O.round_to_kdt(x, "bf16") == one + 2.0 ** -7


def test_bf16_facts_printed_on_vortex_page():
    g = golden("vortex_h2o_constants.txt")
    decay = float(g["default_decay"])
    assert O.round_to_kdt(decay, "bf16") == decay == 1 - 2 ** -6
    # the accumulator climbs to 8.0 from below, where the bf16 spacing is 2^-5
    below8 = float(O.round_to_kdt(7.96875, "bf16"))
    assert below8 < 8.0 and O.ulp_kdt(below8, "bf16") == float(g["bf16_ulp_near_8"])
    inc = float(g["typical_increment"])
    assert inc < 0.5 * float(g["bf16_ulp_near_8"])
    assert O.round_to_kdt(below8 + inc, "bf16") == below8         # the increment is lost
    assert O.round_to_kdt(8.0 + inc, "bf16") == 8.0
    assert abs(O.default_scale(int(g["head_dim"])) - float(g["resolved_scale"])) < 5e-7
    assert 1.0 / (1.0 - decay) == float(g["steady_state_mass"])


# ---------------------------------------------------------------------------
# A1 page statistics
# ---------------------------------------------------------------------------
def _exact_rne(fr: Fraction, p=8, emin=-126):
    """Exact-rational round-to-nearest-even onto a binary grid (independent of numpy)."""
    if fr == 0:
        return 0.0
    a = abs(fr)
    E = math.floor(math.log2(a))
    while Fraction(2) ** E > a:
        E -= 1
    while Fraction(2) ** (E + 1) <= a:
        E += 1
    E = max(E, emin)
    quantum = Fraction(2) ** (E - (p - 1))
    r = round(fr / quantum) * quantum      # Python rounds Fractions half to even
    return float(r)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_page_stats_brute_force(dtype):
    rng = np.random.default_rng(4)
    p, emin = (8, -126) if dtype == "bf16" else (11, -14)
    for f in (1, 2, 3, 7, 16):
        k = O.decode_kdt(O.encode_kdt(rng.standard_normal((f, 24)) * 2.0, dtype), dtype)
        mn, mx, me = O.page_stats(k, dtype)
        for d in range(24):
            col = [float(v) for v in k[:, d]]
            assert mn[d] == min(col) and mx[d] == max(col)
            exact = sum(Fraction(v) for v in col) / f
            assert me[d] == _exact_rne(exact, p, emin)
        if f == 1:
            assert np.array_equal(mn, k[0]) and np.array_equal(mx, k[0]) and np.array_equal(me, k[0])


def test_cache_meta_ignores_positions_past_length():
    rng = np.random.default_rng(5)
    bits = O.encode_kdt(rng.standard_normal((37, 2, 8)), "bf16")
    poisoned = bits.copy()
    poisoned[37 - 5:] = 0x7FC0                    # NaN past a shorter length
    a = O.cache_meta(bits, 32, 16, "bf16")
    b = O.cache_meta(poisoned, 32, 16, "bf16")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    mn, mx, me = O.cache_meta(bits, 37, 16, "bf16")
    assert mn.shape == (3, 2, 8)
    tail = O.decode_kdt(bits[32:37], "bf16")
    assert np.array_equal(mn[2], tail.min(0)) and np.array_equal(mx[2], tail.max(0))


# ---------------------------------------------------------------------------
# A2 page scores
# ---------------------------------------------------------------------------
def test_head_meta_is_cache_meta_of_one_head_and_brute_force():
    """head_meta over one KV head's rows equals that head's slice of
    cache_meta, and both equal min / max / once-rounded mean of each page's
    valid rows taken directly (a partial tail page included)."""
    rng = np.random.default_rng(19)
    for dtype in ("bf16", "fp16"):
        L, H, D, ps = 53, 3, 8, 16
        bits = O.encode_kdt(rng.standard_normal((L + 7, H, D)) * 3, dtype)   # rows past L are stale
        mn, mx, me = O.cache_meta(bits, L, ps, dtype)
        x = O.decode_kdt(bits, dtype)
        for h in range(H):
            hm = O.head_meta(bits[:, h, :], L, ps, dtype)
            for a, c in zip(hm, (mn, mx, me)):
                assert np.array_equal(a, c[:, h, :])
            for p in range(4):
                rows = x[p * ps:min((p + 1) * ps, L), h, :]
                assert np.array_equal(hm[0][p], np.min(rows, axis=0))
                assert np.array_equal(hm[1][p], np.max(rows, axis=0))
                # the exact sum / f rounded once (round_to_kdt is pinned above)
                assert np.array_equal(hm[2][p], O.round_to_kdt(rows.sum(0) / rows.shape[0], dtype))
        assert mn.shape == (4, H, D)


def test_envelope_bounds_true_max_per_head_and_group():
    rng = np.random.default_rng(6)
    for _ in range(200):
        f = int(rng.integers(1, 17))
        G = int(rng.integers(1, 9))
        k = rng.standard_normal((f, 16)) + rng.standard_normal(16)
        q = rng.standard_normal((G, 16))                    # signed queries
        mn, mx = k.min(0), k.max(0)
        s = O.score_pages(mn[None], mx[None], np.zeros((1, 16)), q, 0.0, 1.0)[0]
        true_max = (q @ k.T).max(1)                          # per head, brute force
        per_head = np.array([O.score_pages(mn[None], mx[None], np.zeros((1, 16)), q[g:g + 1], 0.0, 1.0)[0]
                             for g in range(G)])
        assert np.all(per_head >= true_max - 1e-12)
        assert s >= true_max.mean() - 1e-12
        assert abs(s - per_head.mean()) < 1e-12


def test_envelope_is_tight_for_single_token_and_equal_keys():
    rng = np.random.default_rng(7)
    for f in (1, 5):
        row = rng.standard_normal(32)
        k = np.repeat(row[None], f, 0)
        q = rng.standard_normal((3, 32))
        s = O.score_pages(k.min(0)[None], k.max(0)[None], np.zeros((1, 32)), q, 0.0, 1.0)[0]
        assert abs(s - (q @ row).mean()) < 1e-12


def test_average_term_is_mean_attention_logit():
    # integer keys and f = 16: the page mean is exact in bf16, so
    # q . mean(k) = (1/f) sum_j q . k_j exactly up to float64 rounding.
    rng = np.random.default_rng(8)
    k = rng.integers(-8, 9, size=(16, 32)).astype(np.float64)
    q = rng.standard_normal((4, 32))
    mn, mx, me = O.page_stats(k, "bf16")
    s = O.score_pages(mn[None], mx[None], me[None], q, 1.0, 0.0)[0]
    assert abs(s - (q @ k.T).mean()) < 1e-12


def test_linearised_form_equals_plain_form():
    # max(q*M, q*m) = q+ * M + q- * m when M >= m, so the group score equals
    # sum_d [w_avg qbar_d mean_d + w_peak (P_d M_d + N_d m_d)].
    rng = np.random.default_rng(9)
    n, G, D = 50, 8, 64
    k = rng.standard_normal((n, 16, D))
    mn, mx, me = k.min(1), k.max(1), k.mean(1)
    q = rng.standard_normal((G, D))
    s = O.score_pages(mn, mx, me, q, 0.7, 0.3)
    P, N, qb = np.maximum(q, 0).mean(0), np.minimum(q, 0).mean(0), q.mean(0)
    lin = 0.7 * me @ qb + 0.3 * (mx @ P + mn @ N)
    assert np.allclose(s, lin, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# A3 selection
# ---------------------------------------------------------------------------
def _brute_select(s, n, topk):
    if n <= topk:
        return list(range(n))
    cand = list(range(n - 1))

    def better(x, y):  # x ranks strictly before y
        sx, sy = s[x], s[y]
        nx, ny = math.isnan(sx), math.isnan(sy)
        if nx != ny:
            return ny
        if not nx and sx != sy:          # -0.0 == 0.0 in Python
            return sx > sy
        return x < y

    sols = []
    for X in itertools.combinations(cand, topk - 1):
        Xs = set(X)
        if all(better(x, y) for x in Xs for y in cand if y not in Xs):
            sols.append(sorted(X) + [n - 1])
    assert len(sols) == 1
    return sols[0]


def test_select_brute_force_with_ties_zeros_nans():
    rng = np.random.default_rng(10)
    pool = np.array([0.0, -0.0, 1.0, 1.0, -1.0, np.nan, -np.inf, np.inf, 0.5, 0.5, 2.0])
    for _ in range(300):
        n = int(rng.integers(1, 10))
        topk = int(rng.integers(1, 8))
        s = rng.choice(pool, size=n)
        got = O.select_pages(s, n, topk).tolist()
        assert got == _brute_select(list(s), n, topk)


def test_select_edges():
    assert O.select_pages(np.zeros(0), 0, 4).tolist() == []
    assert O.select_pages(np.array([5.0, 1.0, 3.0]), 3, 1).tolist() == [2]       # tail only
    assert O.select_pages(np.array([5.0, 1.0, 3.0]), 3, 3).tolist() == [0, 1, 2]
    assert O.select_pages(np.array([5.0, 1.0, 3.0, 9.0]), 4, 2).tolist() == [0, 3]
    # the tail's own score is irrelevant
    assert O.select_pages(np.array([1.0, 2.0, 3.0, -99.0]), 4, 2).tolist() == [2, 3]


def _brute_select_reserved(s, n, topk, bos, eos):
    """Reserved pages plus the unique window subset every member of which
    ranks before every non-member (score desc, index asc, NaN last)."""
    if n <= topk:
        return list(range(n))
    window = list(range(bos, n - eos))

    def better(x, y):
        sx, sy = s[x], s[y]
        nx, ny = math.isnan(sx), math.isnan(sy)
        if nx != ny:
            return ny
        if not nx and sx != sy:
            return sx > sy
        return x < y

    sols = []
    for X in itertools.combinations(window, topk - bos - eos):
        Xs = set(X)
        if all(better(x, y) for x in Xs for y in window if y not in Xs):
            sols.append(sorted(list(range(bos)) + list(X) + list(range(n - eos, n))))
    assert len(sols) == 1
    return sols[0]


def test_select_reserved_brute_force():
    rng = np.random.default_rng(11)
    pool = np.array([0.0, -0.0, 1.0, 1.0, -1.0, np.nan, -np.inf, np.inf, 0.5, 0.5, 2.0])
    for _ in range(400):
        n = int(rng.integers(1, 11))
        bos = int(rng.integers(0, 3))
        eos = int(rng.integers(1, 3))
        topk = int(rng.integers(bos + eos, bos + eos + 5))
        s = rng.choice(pool, size=n)
        got = O.select_pages_reserved(s, n, topk, bos, eos).tolist()
        assert got == _brute_select_reserved(list(s), n, topk, bos, eos)


def test_select_reserved_reduces_to_tail_forcing():
    rng = np.random.default_rng(12)
    for _ in range(100):
        n = int(rng.integers(1, 300))
        topk = int(rng.integers(1, 40))
        s = rng.standard_normal(n)
        s[rng.random(n) < 0.1] = 0.5
        assert np.array_equal(O.select_pages_reserved(s, n, topk, 0, 1), O.select_pages(s, n, topk))


# ---------------------------------------------------------------------------
# A4 attention and the LSE merge
# ---------------------------------------------------------------------------
def test_attention_matches_library_sdpa():
    from scipy.special import logsumexp
    rng = np.random.default_rng(11)
    for G, n, D in ((1, 1, 8), (4, 37, 64), (8, 300, 128), (3, 17, 128)):
        q, k, v = rng.standard_normal((G, D)), rng.standard_normal((n, D)), rng.standard_normal((n, D))
        sc = D ** -0.5
        o, lse, z = O.attention(q, k, v, sc)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, :, None, :], torch.from_numpy(k)[None, None].expand(1, G, n, D),
            torch.from_numpy(v)[None, None].expand(1, G, n, D), scale=sc)[0, :, 0, :].numpy()
        assert np.allclose(o, ref, rtol=0, atol=1e-12)
        assert np.allclose(lse, logsumexp(sc * q @ k.T, axis=1), rtol=0, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(12)
    q, k, v = rng.standard_normal((4, 16)), rng.standard_normal((1, 16)), rng.standard_normal((1, 16))
    o, lse, _ = O.attention(q, k, v, 0.25)
    assert np.array_equal(o, np.repeat(v, 4, 0))
    assert np.allclose(lse, 0.25 * (q @ k[0]))
    kk = np.repeat(k, 9, 0)
    vv = rng.standard_normal((9, 16))
    o, lse, _ = O.attention(q, kk, vv, 0.25)
    assert np.allclose(o, np.repeat(vv.mean(0, keepdims=True), 4, 0), atol=1e-14)
    assert np.allclose(lse, 0.25 * (q @ k[0]) + math.log(9))
    o, lse, _ = O.attention(q, np.zeros((0, 16)), np.zeros((0, 16)), 0.25)
    assert np.array_equal(o, np.zeros((4, 16))) and np.all(lse == -np.inf)


@pytest.mark.parametrize("S", [1, 2, 3, 7, 16, 200])
def test_chunked_merge_equals_single_shot(S):
    rng = np.random.default_rng(13)
    G, n, D = 8, 200, 64
    q, k, v = rng.standard_normal((G, D)), rng.standard_normal((n, D)) * 2, rng.standard_normal((n, D))
    full_o, full_lse, _ = O.attention(q, k, v, D ** -0.5)
    bounds = np.linspace(0, n, S + 1).astype(int)
    parts = [O.attention(q, k[a:b], v[a:b], D ** -0.5) for a, b in zip(bounds[:-1], bounds[1:])]
    o, lse = O.merge_partials([p[0] for p in parts], [p[1] for p in parts])
    assert np.allclose(o, full_o, atol=1e-12) and np.allclose(lse, full_lse, atol=1e-12)


def test_merge_edge_cases_from_vllmcpp_construction():
    g = golden("vllmcpp_merge_edge_cases.txt")
    T, H, Dm = int(g["tokens"]), int(g["heads"]), int(g["dim"])
    rng = np.random.default_rng(14)
    p_out = rng.uniform(-1, 1, (T, H, Dm))
    s_out = rng.uniform(-1, 1, (T, H, Dm))
    i = np.arange(H * T).reshape(H, T)
    p_lse = (i % 7) * 0.5 - 1.0
    s_lse = (i % 5) * 0.25 + 0.125
    expect = {}
    for c in g["case"]:
        parts = c.split()
        t, h = int(parts[0]), int(parts[1])
        kv = dict(x.split("=") for x in parts[2:])
        if kv["prefix"] != "keep":
            p_lse[h, t] = float(kv["prefix"].replace("+inf", "inf"))
        if kv["suffix"] != "keep":
            s_lse[h, t] = float(kv["suffix"].replace("+inf", "inf"))
        expect[(t, h)] = kv["expect"]
    for t in range(T):
        for h in range(H):
            o, lse = O.merge_partials(np.stack([p_out[t, h][None], s_out[t, h][None]]),
                                      np.array([[p_lse[h, t]], [s_lse[h, t]]]))
            e = expect.get((t, h))
            if e == "suffix":
                assert np.allclose(o[0], s_out[t, h], atol=1e-15) and lse[0] == s_lse[h, t]
            elif e == "prefix":
                assert np.array_equal(o[0], p_out[t, h]) and lse[0] == -np.inf
            else:
                # both finite: the merge weights are a softmax over the two lse
                w = 1.0 / (1.0 + math.exp(s_lse[h, t] - p_lse[h, t]))
                assert np.allclose(o[0], w * p_out[t, h] + (1 - w) * s_out[t, h], atol=1e-14)
                assert abs(lse[0] - np.logaddexp(p_lse[h, t], s_lse[h, t])) < 1e-14


def test_page_decode_all_pages_is_dense_attention():
    # topk >= n_pages selects every page, so the unit equals dense attention
    # over all L cached tokens (textbook routine).
    rng = np.random.default_rng(15)
    L, D, G, ps = 75, 64, 4, 16
    kb = O.encode_kdt(rng.standard_normal((L, D)), "bf16")
    vb = O.encode_kdt(rng.standard_normal((L, D)), "bf16")
    qb = O.encode_kdt(rng.standard_normal((G, D)), "bf16")
    r = O.page_decode_unit(kb, vb, L, qb, ps=ps, topk=100, w_avg=1, w_peak=0.25, dtype="bf16")
    assert r["sel"].tolist() == list(range(5))
    q, k, v = (O.decode_kdt(x, "bf16") for x in (qb, kb, vb))
    ref = torch.softmax(torch.from_numpy(D ** -0.5 * q @ k.T), 1).numpy() @ v
    assert np.allclose(r["out"], ref, atol=1e-12)


# ---------------------------------------------------------------------------
# paged addressing
# ---------------------------------------------------------------------------
def test_reverse_interleaved_table_matches_vllmcpp_construction():
    from sa_synth import reverse_interleaved
    want = np.loadtxt(__import__("os").path.join(
        __import__("os").path.dirname(__file__), "golden", "vllmcpp_reverse_interleaved_3x8.txt"),
        dtype=np.int64, comments="#")
    assert np.array_equal(reverse_interleaved(3, 8, 24), want)


@pytest.mark.parametrize("table", ["reverse", "shuffle", "contiguous"])
def test_gather_through_any_table_recovers_logical_rows(table):
    from sa_synth import reverse_interleaved, shuffled_table, contiguous_table
    rng = np.random.default_rng(16)
    B, H, D, ps, L = 3, 2, 8, 4, 30
    maxp = 8
    NB = B * maxp + 5
    if table == "reverse":
        bt = reverse_interleaved(B, maxp, NB)
    elif table == "shuffle":
        bt = shuffled_table(B, maxp, [maxp] * B, NB, rng)
    else:
        bt = contiguous_table(B, maxp)
    seqs = rng.integers(0, 60000, size=(B, L, H, D)).astype(np.uint16)
    pool = np.full((NB, H, ps, D), 0x7FC0, dtype=np.uint16)
    for b in range(B):
        for j in range(L):
            pool[bt[b, j // ps], :, j % ps] = seqs[b, j]
    for b in range(B):
        for h in range(H):
            rows = O.gather_rows(pool, bt[b], np.arange(L), h, ps)
            assert np.array_equal(rows, seqs[b, :, h])


# ---------------------------------------------------------------------------
# A5 H2O accumulate
# ---------------------------------------------------------------------------
def test_probabilities_sum_to_one_and_decay_one_is_plain_sum():
    from scipy.special import logsumexp
    rng = np.random.default_rng(17)
    z = rng.standard_normal((4, 50)) * 3
    lse = logsumexp(z, axis=1)
    hh0 = np.zeros(50)
    p = O.h2o_fold(hh0, z, lse, 0.5)
    assert abs(p.sum() - 1.0) < 1e-12
    hh = rng.random(50)
    assert np.array_equal(O.h2o_fold(hh, z, lse, 1.0), hh + p)


def test_window_fold_normalises_over_the_window_only():
    rng = np.random.default_rng(19)
    z = rng.standard_normal((4, 40)) * 2
    hh = rng.random(40)
    out = O.h2o_fold_window(hh, z, 3, 5, 0.75)
    p = out - 0.75 * hh
    assert np.all(p[:3] == 0) and np.all(p[-5:] == 0)         # reserved entries receive nothing
    assert abs(p[3:-5].sum() - 1.0) < 1e-12                   # the window's mass is one step's
    # equal logits in the window: each window entry gets 1 / |window| whatever the rest holds
    z2 = z.copy()
    z2[:, 3:-5] = 1.25
    p2 = O.h2o_fold_window(np.zeros(40), z2, 3, 5, 0.5)
    assert np.allclose(p2[3:-5], 1.0 / 32, rtol=0, atol=1e-15)


def test_window_fold_without_reserved_entries_is_the_plain_fold():
    from scipy.special import logsumexp
    rng = np.random.default_rng(20)
    z = rng.standard_normal((3, 25))
    hh = rng.random(25)
    assert np.allclose(O.h2o_fold_window(hh, z, 0, 0, 0.9), O.h2o_fold(hh, z, logsumexp(z, axis=1), 0.9),
                       rtol=1e-14, atol=1e-15)


def test_decayed_mass_closed_form():
    from scipy.special import logsumexp
    rng = np.random.default_rng(18)
    for decay in (0.984375, 0.5, 1.0):
        hh = np.zeros(40)
        T = 300
        for t in range(T):
            z = rng.standard_normal((4, 40))
            hh = O.h2o_fold(hh, z, logsumexp(z, axis=1), decay)
        closed = T if decay == 1.0 else (1 - decay ** T) / (1 - decay)
        assert abs(hh.sum() - closed) < 1e-9 * closed


def _vortex_recurrence(decay, steps, probs):
    hh = np.zeros(probs.shape[1])
    exact = np.zeros(probs.shape[1])
    d = float(O.round_to_kdt(decay, "bf16"))
    for s in range(steps):
        z = np.log(probs[s])[None]                    # log-probs as logits, lse = 0
        hh = O.h2o_store(O.h2o_fold(hh, z, np.zeros(1), d))
        exact = probs[s] + d * exact
    return hh, exact


def test_bf16_accumulator_tracks_exact_recurrence_as_the_vortex_check():
    g = golden("vortex_h2o_constants.txt")
    n, T = int(g["recurrence_tokens"]), int(g["recurrence_steps"])
    rng = np.random.default_rng(19)
    aff = rng.standard_normal(n) * float(g["recurrence_affinity_scale"])
    logits = aff[None] + rng.standard_normal((T, n)) * float(g["recurrence_noise_scale"])
    probs = np.exp(logits - logits.max(1, keepdims=True))
    probs /= probs.sum(1, keepdims=True)
    k = int(g["recurrence_topk"])
    hh, ex = _vortex_recurrence(float(g["default_decay"]), T, probs)
    rel = np.abs(hh - ex).max() / np.abs(ex).max()
    assert rel < float(g["recurrence_rel_err_max"])
    srt = np.sort(ex)[::-1]
    gap, ulp = srt[k - 1] - srt[k], O.ulp_kdt(srt[k - 1], "bf16")
    if gap > ulp:
        assert set(np.argsort(-hh, kind="stable")[:k]) == set(np.argsort(-ex, kind="stable")[:k])
    assert hh.max() < float(g["recurrence_max_bound"])
    probs2 = probs.copy()
    probs2[-1] = 1.0 / n
    hh2, _ = _vortex_recurrence(float(g["default_decay"]), T, probs2)
    assert np.abs(hh - hh2).max() > float(g["recurrence_response_min"])
    # the undecayed bf16 sum freezes and fails the page's own bar
    hh1, ex1 = _vortex_recurrence(1.0, T, probs)
    assert np.abs(hh1 - ex1).max() / np.abs(ex1).max() >= float(g["oracle_final_rel_err_fail"])


# ---------------------------------------------------------------------------
# A5 H2O eviction
# ---------------------------------------------------------------------------
def _bulk_evict(hh, pos, budget, n_sink, grace):
    """Independent characterisation: the m = |R| - budget smallest (score, position)
    pairs among list indices [n_sink, |R| - grace) leave."""
    n = len(pos)
    m = max(0, n - budget)
    elig = sorted(range(n_sink, n - grace), key=lambda j: (hh[j], pos[j]))
    gone = set(elig[:m])
    return [pos[j] for j in range(n) if j not in gone], sorted(pos[j] for j in gone)


def test_evict_matches_bulk_characterisation_with_ties():
    rng = np.random.default_rng(20)
    for _ in range(300):
        n = int(rng.integers(9, 60))
        n_sink, grace = int(rng.integers(0, 4)), int(rng.integers(0, 5))
        budget = int(rng.integers(n_sink + grace + 1, n + 3))
        pos = np.sort(rng.choice(1000, size=n, replace=False))
        hh = rng.choice([0.0, 0.25, 0.5, 0.5, 1.0, 0.125], size=n)
        kept, kept_hh, ev = O.h2o_evict(hh, pos, budget, n_sink, grace)
        bk, bev = _bulk_evict(list(hh), list(pos), budget, n_sink, grace)
        assert kept.tolist() == bk and sorted(ev) == bev
        assert len(kept) == min(n, budget)
        assert np.all(np.diff(kept) > 0)
        assert kept[:n_sink].tolist() == pos[:n_sink].tolist()       # sinks survive
        if grace:
            assert kept[-grace:].tolist() == pos[-grace:].tolist()   # grace survives
        idx = {p: j for j, p in enumerate(pos)}
        assert np.array_equal(kept_hh, hh[[idx[p] for p in kept]])  # untouched values identical


def test_evict_rules_from_velox_evidence():
    pos = np.arange(10)
    hh = np.array([0.0, 0.0, 5, 4, 3, 2, 1, 0.5, 0.0, 0.0])
    # budget + 1 -> exactly budget; sinks survive although they hold the minimum
    kept, _, ev = O.h2o_evict(hh, pos, 9, 2, 0)
    assert len(kept) == 9 and ev == [8]
    # grace protects the newest even when they hold the lowest score
    kept, _, ev = O.h2o_evict(hh, pos, 9, 2, 2)
    assert ev == [7]
    # n_sink = 0: everything is eligible
    kept, _, ev = O.h2o_evict(hh, pos, 9, 0, 0)
    assert ev == [0]
    # tie -> lowest position
    kept, _, ev = O.h2o_evict(np.array([1.0, 0.5, 0.5, 0.5]), np.array([3, 7, 9, 12]), 3, 0, 0)
    assert ev == [7]
    with pytest.raises(ValueError):
        O.h2o_evict(np.zeros(5), np.arange(5), 3, 2, 2)


def test_h2o_unit_step_mass_without_eviction():
    # Each step injects probability mass 1 (new tokens enter at 0), so without
    # eviction the float64 mass after T steps is (1 - decay^T) / (1 - decay).
    g = golden("vortex_h2o_constants.txt")
    decay = float(g["default_decay"])
    rng = np.random.default_rng(21)
    D, G, L0, T = 32, 4, 20, 120
    K = O.encode_kdt(rng.standard_normal((L0 + T, D)), "bf16")
    V = O.encode_kdt(rng.standard_normal((L0 + T, D)), "bf16")
    pos = list(range(L0))
    hh_exact = np.zeros(L0)
    for t in range(T):
        pos.append(L0 + t)
        hh_exact = np.append(hh_exact, 0.0)
        q = O.encode_kdt(rng.standard_normal((G, D)), "bf16")
        r = O.h2o_unit_step(O.h2o_store(hh_exact), pos, K, V, q, dtype="bf16", decay=decay,
                            budget=10 ** 6, n_sink=4, grace=16)
        assert r["kept"].tolist() == pos and r["evicted"] == []
        hh_exact = O.h2o_fold(hh_exact, r["logits"], r["lse"], decay)
    closed = (1 - decay ** T) / (1 - decay)
    assert abs(hh_exact.sum() - closed) < 1e-9


# ---------------------------------------------------------------------------
# N2 H2O with the key as the query (prefill-side absorb and eviction)
# ---------------------------------------------------------------------------
def _batched_absorb(K, decay, scale):
    """The below-budget absorb as one masked matrix product: token i's key
    attends to keys 0..i-1, rows weighted by decay^(T-1-i) and summed."""
    T = K.shape[0]
    Z = (K @ K.T) * scale
    Z[np.triu_indices(T)] = -np.inf                # j >= i is not stored yet
    P = np.zeros_like(Z)
    for i in range(1, T):
        z = Z[i, :i]
        e = np.exp(z - z.max())
        P[i, :i] = e / e.sum()
    w = decay ** (T - 1 - np.arange(T))
    return (w[:, None] * P).sum(axis=0)


def test_proxy_absorb_equals_batched_matrix_form():
    rng = np.random.default_rng(31)
    for decay in (1.0, 0.98, 0.5):
        K = rng.standard_normal((40, 16))
        _, pos, hh, ev = O.h2o_proxy_prefill(K, np.arange(40), decay=decay, budget=100, n_sink=4,
                                             grace=8, scale=0.25, store=False)
        assert ev == [] and pos.tolist() == list(range(40))
        assert np.allclose(hh, _batched_absorb(K, decay, 0.25), rtol=1e-12, atol=1e-14)


def test_proxy_mass_closed_form():
    rng = np.random.default_rng(32)
    T, decay = 60, 0.9
    _, _, hh, _ = O.h2o_proxy_prefill(rng.standard_normal((T, 8)), np.arange(T), decay=decay,
                                      budget=1000, n_sink=0, grace=0, scale=1.0, store=False)
    assert abs(hh.sum() - (1 - decay ** (T - 1)) / (1 - decay)) < 1e-12


def test_proxy_eviction_invariants_and_ties():
    rng = np.random.default_rng(33)
    budget, n_sink, grace = 12, 2, 3
    keys, pos, hh = np.zeros((0, 8)), np.zeros(0, np.int64), np.zeros(0)
    for t in range(80):
        k = rng.standard_normal(8) if t % 7 else np.zeros(8)      # some all-equal attention rows
        before = pos.copy()
        keys, pos, hh, ev = O.h2o_proxy_token(keys, pos, hh, k, t, decay=0.984375, budget=budget,
                                              n_sink=n_sink, grace=grace, scale=0.5)
        assert len(pos) == min(t + 1, budget)
        assert np.all(np.diff(pos) > 0)
        assert pos[:n_sink].tolist() == list(range(min(n_sink, t + 1)))
        assert pos[-grace:].tolist() == list(range(max(0, t + 1 - grace), t + 1))
        if ev is not None:
            # the evicted entry had the minimum stored score among the eligible, lowest position first
            full = np.append(before, t)
            assert ev in full[n_sink:len(full) - grace]
        assert np.all(hh >= 0)


# ---------------------------------------------------------------------------
# N3 alpha-entmax
# ---------------------------------------------------------------------------
def test_sparsemax_worked_example():
    # sorted [1, 0.5, -1]: k = 2 (1 + 2 * 0.5 > 1.5, 1 + 3 * (-1) < 0.5), tau = (1.5 - 1) / 2
    p = O.entmax(np.array([0.5, -1.0, 1.0]), 2.0)
    assert np.allclose(p, [0.25, 0.0, 0.75], atol=1e-15)


def test_entmax15_two_way_closed_form():
    # a = z/2; for two entries in the support, (a1-t)^2 + (a2-t)^2 = 1
    for gap in (0.0, 0.3, 1.0):
        z = np.array([0.0, -gap])
        p = O.entmax(z, 1.5)
        a1, a2 = 0.0, -gap / 2
        t = ((a1 + a2) - np.sqrt((a1 + a2) ** 2 - 2 * (a1 * a1 + a2 * a2 - 1))) / 2
        assert np.allclose(p, [(a1 - t) ** 2, (a2 - t) ** 2], atol=1e-14)
    assert np.allclose(O.entmax(np.array([0.0, -3.0]), 1.5), [1.0, 0.0])   # gap past the support


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_entmax_sort_form_equals_bisection_and_sums_to_one(alpha):
    rng = np.random.default_rng(int(alpha * 10))
    r = 1.0 / (alpha - 1.0)
    for _ in range(50):
        z = rng.standard_normal(int(rng.integers(1, 300))) * rng.choice([0.1, 1.0, 5.0])
        tau = O.entmax_threshold(z, alpha)
        # bisection on the monotone sum, written independently of the sort form
        a = (alpha - 1) * z
        lo, hi = a.max() - 1, a.max()
        for _ in range(200):
            mid = (lo + hi) / 2
            if (np.maximum(a - mid, 0) ** r).sum() >= 1:
                lo = mid
            else:
                hi = mid
        assert abs(tau - (lo + hi) / 2) < 1e-12
        assert abs(O.entmax(z, alpha).sum() - 1.0) < 1e-12


def test_entmax_special_cases():
    for alpha in (1.5, 2.0):
        assert np.allclose(O.entmax(np.zeros(7), alpha), np.full(7, 1 / 7))      # equal logits: uniform
        assert np.allclose(O.entmax(np.array([10.0, 0.0, -1.0]), alpha), [1, 0, 0])
        p = O.entmax(np.array([1.0, -np.inf, 0.9]), alpha)                      # -inf never enters
        assert p[1] == 0 and abs(p.sum() - 1) < 1e-12
    # alpha -> 1 approaches the softmax (bisection path)
    z = np.array([0.3, -0.2, 1.1, 0.0])
    sm = np.exp(z - z.max()); sm /= sm.sum()
    assert np.allclose(O.entmax(z, 1.001), sm, atol=5e-3)


def test_attention_entmax_by_hand_with_a_non_unit_scale():
    """Two query rows, three keys, scale 1/2, every product worked out by hand.

    Row 0: q = (1, 2); q.k = (1, 2, -3), z = (0.5, 1, -1.5). Sparsemax
    (alpha 2): sorted (1, 0.5, -1.5), support 2 (1 + 2 * 0.5 > 1.5,
    1 + 3 * -1.5 < 0.5... gives tau = (1 + 0.5 - 1) / 2 = 0.25), p = (0.25,
    0.75, 0), o = 0.25 * (4, 0) + 0.75 * (0, 8) = (1, 6).
    Row 1: q = (0, 0): equal logits, p = 1/3 each, tau = 0 - 1/3.
    Without the scale row 0 would give tau = 1, p = (0, 1, 0), o = (0, 8);
    with q and k swapped in the product the shapes would not even agree."""
    q = np.array([[1.0, 2.0], [0.0, 0.0]])
    k = np.array([[1.0, 0.0], [0.0, 1.0], [-1.0, -1.0]])
    v = np.array([[4.0, 0.0], [0.0, 8.0], [100.0, 100.0]])
    o, tau, z = O.attention_entmax(q, k, v, 0.5, 2.0)
    assert np.array_equal(z, [[0.5, 1.0, -1.5], [0.0, 0.0, 0.0]])
    assert np.allclose(o[0], [1.0, 6.0], atol=1e-15) and abs(tau[0] - 0.25) < 1e-15
    assert np.allclose(o[1], v.mean(0), atol=1e-13) and abs(tau[1] + 1.0 / 3.0) < 1e-15
    # 1.5-entmax of two keys: a = z / 2 = (q.k) / 4; with q.k = (2, 0),
    # a = (0.5, 0); both in the support iff (a1 - t)^2 + (a2 - t)^2 = 1 has
    # its root t below a2 = 0: t = (0.5 - sqrt(0.25 - 2 * (0.25 - 1))) / 2
    # = (0.5 - sqrt(1.75)) / 2 < 0, so p = ((0.5 - t)^2, t^2).
    q2 = np.array([[2.0, 0.0]])
    k2 = np.array([[1.0, 3.0], [0.0, -5.0]])
    v2 = np.array([[1.0, 0.0], [0.0, 1.0]])
    o2, tau2, z2 = O.attention_entmax(q2, k2, v2, 0.5, 1.5)
    t = (0.5 - math.sqrt(1.75)) / 2
    assert np.array_equal(z2, [[1.0, 0.0]])
    assert abs(tau2[0] - t) < 1e-15
    assert np.allclose(o2[0], [(0.5 - t) ** 2, t * t], atol=1e-15)
    assert abs((0.5 - t) ** 2 + t * t - 1.0) < 1e-14


def test_page_decode_unit_entmax_with_every_page_is_dense_entmax():
    """All pages selected: the unit's entmax output is entmax attention over
    every cached token, and alpha = 1 keeps the softmax path."""
    rng = np.random.default_rng(21)
    L, D, G, ps = 45, 16, 2, 8
    kb = O.encode_kdt(rng.standard_normal((L, D)), "bf16")
    vb = O.encode_kdt(rng.standard_normal((L, D)), "bf16")
    qb = O.encode_kdt(rng.standard_normal((G, D)), "bf16")
    for alpha in (1.5, 2.0):
        r = O.page_decode_unit(kb, vb, L, qb, ps=ps, topk=99, w_avg=1.0, w_peak=0.25,
                               dtype="bf16", alpha=alpha)
        k, v, q = (O.decode_kdt(x, "bf16") for x in (kb, vb, qb))
        o, tau, _ = O.attention_entmax(q, k, v, D ** -0.5, alpha)
        assert np.array_equal(r["out"], o) and np.array_equal(r["tau"], tau)
        # rows of p sum to 1: o lies in the convex hull of V, per dimension
        assert np.all(r["out"] <= v.max(0) + 1e-12) and np.all(r["out"] >= v.min(0) - 1e-12)
    r1 = O.page_decode_unit(kb, vb, L, qb, ps=ps, topk=99, w_avg=1.0, w_peak=0.25, dtype="bf16")
    assert "lse" in r1


# ---------------------------------------------------------------------------
# N4 Gaussian-aware selection
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_gauss_tail_moment_matches_quadrature(alpha):
    """The truncated-normal closed forms against numerical integration of the
    defining expectation E[((alpha - 1) Z - t)_+^(1/(alpha - 1))]."""
    from scipy import integrate
    r = 1.0 / (alpha - 1.0)
    for mu, sd, t in [(0.0, 1.0, 0.3), (0.7, 0.4, 0.1), (-1.2, 2.5, -0.4), (2.0, 0.3, 1.6),
                      (0.0, 1.0, 2.5)]:
        f = lambda z: max((alpha - 1.0) * z - t, 0.0) ** r * math.exp(-0.5 * ((z - mu) / sd) ** 2) / (sd * math.sqrt(2 * math.pi))
        lo = t / (alpha - 1.0)
        want = integrate.quad(f, lo, mu + 40 * sd, epsabs=1e-14, epsrel=1e-12, limit=200)[0]
        got = O.gauss_tail_moment(mu, sd, t, alpha)
        assert abs(got - want) <= 1e-9 * max(1.0, abs(want)), (mu, sd, t, got, want)
    # no spread: the moment of a point mass
    assert O.gauss_tail_moment(0.9, 0.0, 0.1, alpha) == pytest.approx(((alpha - 1) * 0.9 - 0.1) ** r)
    assert O.gauss_tail_moment(0.1, 0.0, 0.5, alpha) == 0.0


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_gauss_tau_point_mass_and_sample_entmax(alpha):
    # V = 0: N equal scores share the mass, N ((alpha-1) M - tau)^r = 1
    for N, M in [(16, 0.4), (4096, -1.3), (1, 2.0)]:
        want = (alpha - 1.0) * M - N ** (-(alpha - 1.0))
        assert O.gauss_tau(N, M, 0.0, alpha) == pytest.approx(want, abs=1e-12)
    # a large Gaussian sample: the exact entmax threshold of the sample,
    # averaged over draws, agrees with the distributional tau_hat within its
    # standard error
    rng = np.random.default_rng(31)
    N, M, sd, reps = 5000, 0.3, 0.8, 40
    ts = [O.entmax_threshold(M + sd * rng.standard_normal(N), alpha) for _ in range(reps)]
    se = np.std(ts) / math.sqrt(reps)
    assert abs(np.mean(ts) - O.gauss_tau(N, M, sd * sd, alpha)) <= 4 * se
    # more scores push the threshold up
    assert O.gauss_tau(2 * N, M, sd * sd, alpha) > O.gauss_tau(N, M, sd * sd, alpha)


def _hadamard(n):
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def test_gauss_page_moments_exact_on_uncorrelated_pages():
    """Pages whose keys are mean + std * (rows of a Hadamard matrix without
    its constant column): per-dimension mean and population std are exactly
    mean and std, the dimensions are exactly uncorrelated, so the diagonal
    model's page moments are exactly the empirical mean and variance of the
    page's scores, and the mixture moments those of all scores."""
    H = _hadamard(16)[:, 1:]                          # 16 tokens x 15 dims, zero-mean orthogonal columns
    rng = np.random.default_rng(5)
    scale = 0.125
    q = rng.integers(-8, 9, size=15) / 8.0
    pages, ms, vs = [], [], []
    for p in range(5):
        mean = rng.integers(-16, 17, size=15) / 16.0
        std = rng.integers(1, 9, size=15) / 8.0
        keys = mean + std * H                          # exactly representable in bf16
        assert np.array_equal(O.round_to_kdt(keys, "bf16"), keys)
        got_std = O.page_std(keys, "bf16")
        assert np.array_equal(got_std, std) and np.array_equal(keys.mean(0), mean)
        m, v = O.gauss_page_moments(q, mean[None], got_std[None], scale)
        z = scale * keys @ q
        assert m[0] == pytest.approx(z.mean(), rel=1e-12, abs=1e-12)
        assert v[0] == pytest.approx(z.var(), rel=1e-12)
        pages.append(z); ms.append(m[0]); vs.append(v[0])
    N, M, V = O.gauss_global_moments(np.array(ms), np.array(vs), np.full(5, 16))
    allz = np.concatenate(pages)
    assert N == 80 and M == pytest.approx(allz.mean(), abs=1e-12) and V == pytest.approx(allz.var(), rel=1e-12)


def test_gauss_max_factor_bounds_the_expected_maximum():
    # E[max of 2 standard normals] = 1 / sqrt(pi); Monte Carlo for larger f
    assert 1.0 / math.sqrt(math.pi) <= O.gauss_max_factor(2)
    rng = np.random.default_rng(2)
    for f in (3, 8, 16):
        emax = rng.standard_normal((200000, f)).max(1).mean()
        assert emax <= O.gauss_max_factor(f)
    assert O.gauss_max_factor(1) == 0.0


def test_gauss_select_rule():
    m = np.array([0.0, 3.0, -1.0, 0.5, 0.0])
    v = np.array([1.0, 0.0, 0.0, 4.0, 0.0])
    fill = np.array([16, 16, 1, 16, 3])
    # (alpha - 1) * (m + sqrt(2 ln f) sqrt(v)) against tau_hat, tail always
    est = [0 + math.sqrt(2 * math.log(16)), 3.0, -1.0, 0.5 + 2 * math.sqrt(2 * math.log(16)), 0.0]
    for alpha, th in [(2.0, 2.9), (1.5, 1.49), (2.0, 100.0), (2.0, -5.0)]:
        want = [p for p in range(5) if (alpha - 1) * est[p] > th or p == 4]
        assert O.gauss_select(m, v, fill, th, alpha).tolist() == want
    # a higher threshold keeps a subset
    a = set(O.gauss_select(m, v, fill, 0.5, 2.0).tolist())
    b = set(O.gauss_select(m, v, fill, 2.0, 2.0).tolist())
    assert b <= a


def test_gauss_select_against_the_pages_known_maxima():
    """Pages built so the maximum of their scores is known exactly, the
    threshold crossing it: every single-token page and every page of equal
    keys (v = 0) is kept exactly when its one score value is in the entmax
    support at tau_hat ((alpha - 1) z > tau_hat), whatever kappa is; a page of
    two-valued scores (Hadamard rows: scores m +- s, half each, so v = s^2)
    whose top value crosses is always kept (kappa_16 > 1 makes the estimate
    an upper bound of that top value); such a page whose top value stays
    below but whose estimate m + kappa s crosses is kept too (the estimate,
    not the sample, decides), and one whose estimate stays below is dropped.
    The tail (last page) is kept regardless."""
    H = _hadamard(16)[:, 1:2]                             # one +-1 column, 16 tokens
    scale = 0.5
    q = np.array([1.0])
    kap = math.sqrt(2 * math.log(16))
    for alpha in (1.5, 2.0):
        th = 0.8 * (alpha - 1.0)                          # a score z crosses iff z > 0.8
        pages, top, kind = [], [], []
        # single tokens (f = 1): z = scale * key
        for key in (1.2, 1.6, 1.61, -4.0):
            pages.append(np.array([[key]])); top.append(scale * key); kind.append("point")
        # equal keys (f = 16, v = 0)
        for key in (1.0, 2.0):
            pages.append(np.full((16, 1), key)); top.append(scale * key); kind.append("point")
        # two-valued pages: key = c + d * (+-1): m = scale c, s = scale d
        for c_, d_, want in ((1.2, 0.6, "top"), (0.8, 0.5, "est"), (0.0, 0.25, "none")):
            pages.append(c_ + d_ * H); top.append(scale * (c_ + d_)); kind.append(want)
        pages.append(np.array([[-9.0]])); top.append(-4.5); kind.append("tail")
        means = np.array([pg.mean(0) for pg in pages])
        stds = np.array([O.page_std(pg, "bf16") for pg in pages])
        fill = np.array([pg.shape[0] for pg in pages])
        m, v = O.gauss_page_moments(q, means, stds, scale)
        sel = set(O.gauss_select(m, v, fill, th, alpha).tolist())
        n = len(pages)
        for p in range(n):
            crosses = (alpha - 1.0) * top[p] > th
            if kind[p] == "point":
                assert (p in sel) == crosses, (alpha, p, top[p])
            elif kind[p] == "top":
                assert crosses and p in sel
            elif kind[p] == "est":
                assert not crosses and (alpha - 1.0) * (m[p] + kap * math.sqrt(v[p])) > th
                assert p in sel
            elif kind[p] == "none":
                assert (alpha - 1.0) * (m[p] + kap * math.sqrt(v[p])) < th and p not in sel
        assert n - 1 in sel and not (alpha - 1.0) * top[n - 1] > th


def test_gauss_decode_unit_one_page_is_dense_entmax():
    """A request of one page selects it (the tail): the unit is entmax
    attention over every token, with the exact tau of that selection."""
    rng = np.random.default_rng(12)
    L, D = 13, 32
    kb = O.encode_kdt(rng.standard_normal((L, D)), "bf16")
    vb = O.encode_kdt(rng.standard_normal((L, D)), "bf16")
    qb = O.encode_kdt(rng.standard_normal(D), "bf16")
    for alpha in (1.5, 2.0):
        r = O.gauss_decode_unit(kb, vb, L, qb, ps=16, alpha=alpha, dtype="bf16")
        k, v, q = (O.decode_kdt(x, "bf16") for x in (kb, vb, qb))
        o, tau, _ = O.attention_entmax(q[None], k, v, D ** -0.5, alpha)
        assert r["sel"].tolist() == [0]
        assert np.array_equal(r["out"], o[0]) and r["tau"] == tau[0]
