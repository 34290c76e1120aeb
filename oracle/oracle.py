"""CPU oracle for one decode step of page-selected sparse attention over a paged
KV cache, and for the token-level H2O accumulate / evict update.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline / reference leg may import this module. The product path
(package ``sparse_paged_kv_page_gb300``) never imports it and has no CPU
fallback to it. This module imports nothing from the product path either.

Everything here is float64 numpy written as the plain definition: no blocking,
fusion, linearisation or reordering beyond what a definition states. Inputs are
bf16/fp16 *bit patterns* (uint16) and int32 tables, exactly as the seeded
generator produces them; values are decoded to float64 here.

Sources, cited by page title and section:

* [vortex]  "flow: add H2O sparse attention (page-level and token-level, MHA +
            GQA)", vortex_torch pull request 6 -- sections "Page-level
            variants", "Token-level variants", "Verification", and the
            follow-up comment's oracle harness.
* [velox]   "H2O -- Cumulative Attention-Mass Heavy-Hitter Oracle Eviction",
            VeloxQuant-MLX docs -- sections "Parameters", "How it works",
            "Fidelity to Algorithm 1", "Evidence".
* [vllmcpp] "test_ops_mla_chunked_context.cpp", vllm.cpp tests -- the
            double-precision single-shot attention oracle and the
            "MergeAttnStates" LSE edge-case test.
* [entmax]  "EntmaxKV" README -- sections "How it works" (top-k and
            Gaussian-aware strategies), "Quick start".

Readings taken where the pages are silent (each restated where it is used):

* page statistics cover only the f_p valid tokens of a page (stale slots of
  a partially filled tail page are never read);
* the KV-head page score is the mean over the G query heads of the per-head
  scores w_avg*avg + w_peak*peak (the pages say the group is reduced to one
  ranking, not by which operator);
* scores carry no softmax scale (both terms are linear in q);
* selection order is (score descending, page index ascending), -0 == +0,
  NaN after every number; selected indices are returned ascending;
* H2O: the new token attends to itself; p_bar is the mean over the G heads of
  the true softmax probabilities over all retained tokens; the update is
  hh <- decay*hh + p_bar rounded once to bf16; eviction removes, one at a
  time, the minimum-(score, position) entry among list indices
  [n_sink, |R| - grace) while |R| > budget.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

# precision p (significand bits incl. the implicit one), e_min, e_max
_FORMATS = {"bf16": (8, -126, 127), "fp16": (11, -14, 15)}


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def decode_kdt(bits, dtype: str) -> np.ndarray:
    """uint16 bit patterns of bf16 / fp16 -> float64 values (exact)."""
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        if dtype == "bf16":
            return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        if dtype == "fp16":
            return bits.view(np.float16).astype(np.float64)
    raise ValueError(dtype)


def round_to_kdt(x, dtype: str) -> np.ndarray:
    """Round float64 values once, ties to even, onto the bf16 / fp16 grid.

    IEEE 754 roundTiesToEven applied directly to the float64 value (one
    rounding, no intermediate float32): in the binade of x the grid spacing is
    2^(E-(p-1)) with E = max(floor(log2|x|), e_min); values beyond the largest
    finite number round to +-inf.
    """
    p, emin, emax = _FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(x)                       # |x| = m * 2^e, m in [0.5, 1)
        E = np.maximum(e - 1, emin)
        quantum = np.ldexp(1.0, E - (p - 1))
        r = np.rint(x / quantum) * quantum       # np.rint rounds half to even
        maxf = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
        r = np.where(np.abs(r) > maxf, np.copysign(np.inf, x), r)
        r = np.where(np.isfinite(x), r, x)
    return r


def encode_kdt(x, dtype: str) -> np.ndarray:
    """float64 -> uint16 bit patterns (via :func:`round_to_kdt`)."""
    r = round_to_kdt(x, dtype)
    if dtype == "bf16":
        return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return r.astype(np.float16).view(np.uint16)


def ulp_kdt(x, dtype: str) -> np.ndarray:
    """Spacing of the bf16 / fp16 grid at |x| (subnormal spacing below e_min)."""
    p, emin, _ = _FORMATS[dtype]
    _, e = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))
    return np.ldexp(1.0, np.maximum(e - 1, emin) - (p - 1))


# ---------------------------------------------------------------------------
# paged layout
# ---------------------------------------------------------------------------
def num_pages(L: int, ps: int) -> int:
    """Pages holding L tokens; page p holds positions [p*ps, min((p+1)*ps, L))."""
    return -(-int(L) // int(ps))


def page_positions(p: int, L: int, ps: int) -> np.ndarray:
    return np.arange(p * ps, min((p + 1) * ps, L))


def gather_rows(pool_bits, block_table_row, positions, h: int, ps: int) -> np.ndarray:
    """Rows of KV head h at logical positions, read from a paged pool through the
    block table: position j lives in physical block bt[j // ps], slot j % ps.

    pool_bits: uint16 [num_blocks, H_kv, ps, D]: each (block, head) a contiguous ps x D tile.
    [entmax] "How it works": pages in a block-table paged layout.
    """
    positions = np.asarray(positions, dtype=np.int64)
    blk = np.asarray(block_table_row, dtype=np.int64)[positions // ps]
    return pool_bits[blk, h, positions % ps]


# ---------------------------------------------------------------------------
# A1: page statistics
# ---------------------------------------------------------------------------
def page_stats(k_tok: np.ndarray, dtype: str):
    """Element-wise k_min, k_max, k_mean of the f >= 1 valid keys of one page.

    [vortex] "Page-level variants" and "Token-level variants" point 2 (CMin /
    CMax / CMean are overwriting reductions over the page); [entmax] "How it
    works" (per-page key statistics). k_tok: float64 [f, D]. min / max are
    exact; the mean is (1/f) * sum, rounded once to the cache dtype because the
    statistics are stored in it.
    """
    f = k_tok.shape[0]
    assert f >= 1
    return k_tok.min(0), k_tok.max(0), round_to_kdt(k_tok.sum(0) / f, dtype)


def cache_meta(k_seq_bits, L: int, ps: int, dtype: str):
    """Statistics of every page of one request. k_seq_bits: uint16 [L, H_kv, D].

    Returns (k_min, k_max, k_mean), each float64 [n_pages, H_kv, D]."""
    k = decode_kdt(k_seq_bits[:L], dtype)
    n = num_pages(L, ps)
    H, D = k.shape[1], k.shape[2]
    mn = np.empty((n, H, D))
    mx = np.empty((n, H, D))
    me = np.empty((n, H, D))
    for p in range(n):
        rows = k[p * ps:min((p + 1) * ps, L)]              # [f, H, D]
        for h in range(H):
            mn[p, h], mx[p, h], me[p, h] = page_stats(rows[:, h, :], dtype)
    return mn, mx, me


def head_meta(k_head_bits, L: int, ps: int, dtype: str):
    """Statistics of every page of one request for one KV head.

    k_head_bits: uint16 [L, D]. Returns three float64 arrays [n_pages, D]."""
    k = decode_kdt(k_head_bits[:L], dtype)
    n = num_pages(L, ps)
    D = k.shape[1]
    mn, mx, me = np.empty((n, D)), np.empty((n, D)), np.empty((n, D))
    for p in range(n):
        mn[p], mx[p], me[p] = page_stats(k[p * ps:min((p + 1) * ps, L)], dtype)
    return mn, mx, me


# ---------------------------------------------------------------------------
# A2: page scores
# ---------------------------------------------------------------------------
def score_pages(k_min, k_max, k_mean, q, w_avg: float, w_peak: float,
                chunk: int = 2048) -> np.ndarray:
    """KV-head page score of every page.

    [vortex] "Page-level variants": average relevance q . mean(k); peak
    relevance, the envelope bound sum_d max(q_d * max_d, q_d * min_d) >=
    max_k q . k (both envelopes, because q is signed); combined as
    w_avg * avg + w_peak * peak. GQA: the G query heads of a KV head are
    reduced to one ranking, here by the mean of their scores. No softmax scale.

    k_min, k_max, k_mean: float64 [n, D]; q: float64 [G, D]. Returns [n].
    """
    n = k_min.shape[0]
    out = np.empty(n)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        avg = k_mean[s:e] @ q.T                                       # [c, G]
        peak = np.maximum(k_max[s:e, None, :] * q[None, :, :],
                          k_min[s:e, None, :] * q[None, :, :]).sum(-1)  # [c, G]
        out[s:e] = (w_avg * avg + w_peak * peak).mean(1)
    return out


# ---------------------------------------------------------------------------
# A3: top-k with the tail page forced
# ---------------------------------------------------------------------------
def select_pages(scores, n_pages: int, topk: int) -> np.ndarray:
    """Indices of the pages attended, ascending.

    [entmax] "Top-k": keep topk pages; the budget counts pages and includes
    the always-attended tail page n_pages-1. If n_pages <= topk every page is
    kept. Otherwise the tail plus the topk-1 best of pages 0..n_pages-2 by
    (score descending, index ascending); -0 and +0 are equal; NaN ranks after
    every number.
    """
    n_pages = int(n_pages)
    if n_pages <= 0:
        return np.zeros(0, dtype=np.int64)
    if n_pages <= topk:
        return np.arange(n_pages, dtype=np.int64)
    s = np.asarray(scores[:n_pages - 1], dtype=np.float64)
    nan = np.isnan(s)
    key = np.where(nan, 0.0, -s) + 0.0          # +0.0 maps -0 to +0
    idx = np.arange(n_pages - 1)
    order = np.lexsort((idx, key, nan))         # last key is primary
    chosen = np.concatenate([order[:topk - 1], [n_pages - 1]])
    return np.sort(chosen).astype(np.int64)


def select_pages_reserved(scores, n_pages: int, topk: int, n_bos: int, n_eos: int) -> np.ndarray:
    """Indices of the pages attended with reserved leading and trailing pages.

    [vortex] follow-up comment, "Two things I had to fix": the first
    page_reserved_bos and the last page_reserved_eos pages are kept
    unconditionally and top-k only ranks the window between them. Reading: the
    reserved pages count against the budget topk, as [entmax] "Top-k" counts
    the always-attended tail page (n_bos = 0, n_eos = 1 is select_pages). If
    n_pages <= topk every page is kept; otherwise the reserved pages plus the
    topk - n_bos - n_eos best of the window by (score descending, index
    ascending), -0 == +0, NaN last.
    """
    n = int(n_pages)
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    if n <= topk:
        return np.arange(n, dtype=np.int64)
    lo, hi, kk = int(n_bos), n - int(n_eos), topk - int(n_bos) - int(n_eos)
    s = np.asarray(scores[lo:hi], dtype=np.float64)
    nan = np.isnan(s)
    key = np.where(nan, 0.0, -s) + 0.0
    idx = np.arange(lo, hi)
    order = np.lexsort((idx, key, nan))
    chosen = np.concatenate([np.arange(lo), idx[order[:kk]], np.arange(hi, n)])
    return np.sort(chosen).astype(np.int64)


# ---------------------------------------------------------------------------
# N3: alpha-entmax in place of the softmax over the selected tokens
# ---------------------------------------------------------------------------
def entmax_threshold(z, alpha: float) -> float:
    """tau of alpha-entmax: p_i = [(alpha-1) z_i - tau]_+ ** (1/(alpha-1)), sum p = 1.

    [entmax] "How it works" and "Quick start" (alpha = 1.5 by default, 1.5 and
    2 decoded exactly). With a = (alpha - 1) z sorted descending and a support
    of the k largest, sum_{i<=k} (a_i - tau)^(1/(alpha-1)) = 1 fixes tau:
      alpha = 2:   tau = (sum_{i<=k} a_i - 1) / k
      alpha = 1.5: k tau^2 - 2 tau S1 + S2 - 1 = 0, the root below a_k,
    and the support is the largest k whose tau stays below a_k. Other alpha
    by bisection on the monotone sum. -inf entries never enter the support.
    """
    a = np.sort((alpha - 1.0) * np.asarray(z, np.float64)[np.isfinite(z)])[::-1]
    if a.size == 0:
        raise ValueError("no finite logits")
    if alpha == 2.0 or alpha == 1.5:
        S1 = np.cumsum(a)
        S2 = np.cumsum(a * a)
        k = np.arange(1, a.size + 1)
        if alpha == 2.0:
            tau = (S1 - 1.0) / k
        else:
            disc = np.maximum(S1 * S1 - k * (S2 - 1.0), 0.0)
            tau = (S1 - np.sqrt(disc)) / k
        ok = tau < a                                  # every member of the support stays positive
        kk = int(np.nonzero(ok)[0].max())             # largest such k (k = 1 always qualifies)
        return float(tau[kk])
    r = 1.0 / (alpha - 1.0)
    lo, hi = a[0] - 1.0, a[0]
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if (np.maximum(a - mid, 0.0) ** r).sum() >= 1.0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def entmax(z, alpha: float) -> np.ndarray:
    """alpha-entmax probabilities of logits z (see entmax_threshold)."""
    z = np.asarray(z, np.float64)
    tau = entmax_threshold(z, alpha)
    p = np.where(np.isfinite(z), np.maximum((alpha - 1.0) * z - tau, 0.0), 0.0)
    return p ** (1.0 / (alpha - 1.0))


def attention_entmax(q, k, v, scale: float, alpha: float):
    """Attention with alpha-entmax in place of the softmax: for each query row,
    o = sum_j entmax(scale q.k_j)_j v_j. Returns (o [G, D], tau [G], z [G, T])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    z = (q @ k.T) * scale
    o = np.zeros((q.shape[0], v.shape[1]))
    tau = np.full(q.shape[0], np.nan)
    for g in range(q.shape[0]):
        if z.shape[1] == 0:
            continue
        tau[g] = entmax_threshold(z[g], alpha)
        o[g] = entmax(z[g], alpha) @ v
    return o, tau, z


# ---------------------------------------------------------------------------
# N4: Gaussian-aware selection
# ---------------------------------------------------------------------------
def page_std(k_tok: np.ndarray, dtype: str) -> np.ndarray:
    """Element-wise k_std of the f >= 1 valid keys of one page.

    [entmax] "How it works" (mean / std per page for the Gaussian strategy)
    and its k_mean / k_std refresh: the population standard deviation
    sqrt((1/f) sum (k - mean)^2) around the exact mean, rounded once to the
    cache dtype (stored like k_mean). k_tok: float64 [f, D].
    """
    mean = k_tok.mean(0)
    return round_to_kdt(np.sqrt(((k_tok - mean) ** 2).mean(0)), dtype)


def head_gauss_stats(k_head_bits, L: int, ps: int, dtype: str):
    """k_mean, k_std and the fill of every page of one (request, KV head).

    k_head_bits: uint16 [L, D]. Returns float64 [n, D], [n, D], int [n]."""
    k = decode_kdt(k_head_bits[:L], dtype)
    n = num_pages(L, ps)
    me, sd = np.empty((n, k.shape[1])), np.empty((n, k.shape[1]))
    fill = np.empty(n, dtype=np.int64)
    for p in range(n):
        rows = k[p * ps:min((p + 1) * ps, L)]
        me[p] = round_to_kdt(rows.sum(0) / rows.shape[0], dtype)
        sd[p] = page_std(rows, dtype)
        fill[p] = rows.shape[0]
    return me, sd, fill


def gauss_page_moments(q, k_mean, k_std, scale: float):
    """Query-conditioned moments of a page's scores z = scale * q . k.

    [entmax] "How it works" (each page's scores modelled as a Gaussian) and
    its query-conditioned page moments: with the key dimensions of a page
    taken as independent (the statistics are per dimension),
      m_p = scale * sum_d q_d mean_pd,   v_p = scale^2 * sum_d q_d^2 std_pd^2.
    q: [D] (one query head); k_mean, k_std: [n, D]. Returns m, v [n].
    """
    q = np.asarray(q, np.float64)
    return scale * (k_mean @ q), scale * scale * ((k_std ** 2) @ (q * q))


def gauss_global_moments(m, v, fill):
    """Mean and variance of all N = sum f_p scores of the page mixture
    (page p holds f_p scores of mean m_p and variance v_p):
    M = sum f m / N, V = sum f (v + m^2) / N - M^2. The single-Gaussian model
    ([entmax] How it works: heads without ALiBi) is N(M, V)."""
    f = np.asarray(fill, np.float64)
    N = f.sum()
    M = (f * m).sum() / N
    V = max((f * (v + m * m)).sum() / N - M * M, 0.0)
    return N, M, V


def _phi(u):
    return math.exp(-0.5 * u * u) / math.sqrt(2.0 * math.pi)


def _Phi(u):
    return 0.5 * math.erfc(-u / math.sqrt(2.0))


def gauss_tail_moment(mu: float, sigma: float, t: float, alpha: float) -> float:
    """E[((alpha - 1) Z - t)_+ ^ (1 / (alpha - 1))] for Z ~ N(mu, sigma^2),
    alpha in {1.5, 2}: with a = (alpha - 1) Z ~ N(mu_a, s_a^2), c = mu_a - t
    and u = c / s_a, the truncated moments of the normal give
      alpha 2:   c Phi(u) + s_a phi(u)
      alpha 1.5: (c^2 + s_a^2) Phi(u) + c s_a phi(u)
    and ((c)_+)^r when sigma = 0."""
    if alpha not in (1.5, 2.0):
        raise ValueError("closed forms for alpha 1.5 and 2 only")
    mu_a, s_a = (alpha - 1.0) * mu, (alpha - 1.0) * sigma
    c = mu_a - t
    if s_a == 0.0:
        return max(c, 0.0) ** (1.0 / (alpha - 1.0))
    u = c / s_a
    if alpha == 2.0:
        return c * _Phi(u) + s_a * _phi(u)
    return (c * c + s_a * s_a) * _Phi(u) + c * s_a * _phi(u)


def gauss_tau(N: float, M: float, V: float, alpha: float) -> float:
    """tau_hat of the distributional entmax constraint ([entmax] How it works):
    N scores drawn from N(M, V) should carry unit entmax mass,
    N * E[((alpha - 1) Z - tau)_+ ^ (1 / (alpha - 1))] = 1. The left side
    decreases strictly in tau (while positive); bisection on a bracket whose
    ends are checked."""
    sd = math.sqrt(V)
    lo = (alpha - 1.0) * (M + 10.0 * sd) - 1.0
    while N * gauss_tail_moment(M, sd, lo, alpha) < 1.0:
        lo -= 1.0 + abs(lo)
    hi = (alpha - 1.0) * (M + 12.0 * sd) + 1.0
    while N * gauss_tail_moment(M, sd, hi, alpha) > 1.0:
        hi += 1.0 + abs(hi)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if N * gauss_tail_moment(M, sd, mid, alpha) >= 1.0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def gauss_max_factor(f: int) -> float:
    """kappa_f with E[max of f scores] <= m + kappa_f sqrt(v) for f scores of
    mean m and variance v that are jointly Gaussian (any correlation):
    sqrt(2 ln f); 0 for a single token. The pages select every page whose
    estimated maximum can cross tau_hat; this bound is the estimate taken."""
    return math.sqrt(2.0 * math.log(f)) if f > 1 else 0.0


def gauss_select(m, v, fill, tau_hat: float, alpha: float) -> np.ndarray:
    """Pages p with (alpha - 1) * (m_p + kappa_{f_p} sqrt(v_p)) > tau_hat, and
    the tail page always ([entmax] How it works, Top-k: the tail is attended);
    ascending. The count adapts to the distribution; no budget."""
    n = len(m)
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    est = np.array([m[p] + gauss_max_factor(int(fill[p])) * math.sqrt(v[p]) for p in range(n)])
    keep = (alpha - 1.0) * est > tau_hat
    keep[n - 1] = True
    return np.nonzero(keep)[0].astype(np.int64)


def gauss_decode_unit(k_head_bits, v_head_bits, L: int, q_bits, *, ps: int, alpha: float,
                      dtype: str, scale: float = 0.0):
    """N4 for one query head of one request: page k_mean / k_std, the page
    moments of this head's scores, tau_hat of the single Gaussian, threshold
    selection (+ tail), then alpha-entmax attention over the selected pages'
    valid tokens with the exact tau of that selection (the "corrected" tau).

    k_head_bits, v_head_bits: uint16 [L, D] of the head's KV head; q_bits:
    uint16 [D]. Returns dict(mean, std, fill, m, v, N, M, V, tau_hat, sel,
    out [D], tau)."""
    D = k_head_bits.shape[1]
    sc = scale if scale > 0 else default_scale(D)
    q = decode_kdt(q_bits, dtype)
    me, sd, fill = head_gauss_stats(k_head_bits, L, ps, dtype)
    m, v = gauss_page_moments(q, me, sd, sc)
    N, M, V = gauss_global_moments(m, v, fill)
    th = gauss_tau(N, M, V, alpha)
    sel = gauss_select(m, v, fill, th, alpha)
    pos = selected_positions(sel, L, ps)
    k = decode_kdt(k_head_bits[pos], dtype)
    vv = decode_kdt(v_head_bits[pos], dtype)
    o, tau, _ = attention_entmax(q[None, :], k, vv, sc, alpha)
    return {"mean": me, "std": sd, "fill": fill, "m": m, "v": v, "N": N, "M": M, "V": V,
            "tau_hat": th, "sel": sel, "out": o[0], "tau": float(tau[0])}


# ---------------------------------------------------------------------------
# A4: attention over the selected tokens, and the LSE merge
# ---------------------------------------------------------------------------
def default_scale(D: int) -> float:
    """[vortex] "Token-level variants" point 1: the softmax scale defaults to head_dim ** -0.5."""
    return float(D) ** -0.5


def attention(q, k, v, scale: float):
    """Exact softmax attention of G query rows over n keys, two passes.

    Follows the [vllmcpp] double-precision oracle: logits z = scale * q . k_j;
    m = max z; o = sum_j exp(z_j - m) v_j / sum_j exp(z_j - m); and
    lse = m + log sum_j exp(z_j - m). No keys: o = 0, lse = -inf.
    q: [G, D]; k, v: [n, D] float64. Returns o [G, D], lse [G], z [G, n].
    """
    G = q.shape[0]
    n = k.shape[0]
    if n == 0:
        return np.zeros((G, v.shape[1])), np.full(G, -np.inf), np.zeros((G, 0))
    z = scale * (q @ k.T)
    m = z.max(1, keepdims=True)
    e = np.exp(z - m)
    l = e.sum(1)
    o = (e @ v) / l[:, None]
    return o, m[:, 0] + np.log(l), z


def selected_positions(sel_pages, L: int, ps: int) -> np.ndarray:
    """Positions of the valid tokens of the selected pages, ascending."""
    parts = [page_positions(int(p), L, ps) for p in sel_pages]
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def merge_partials(o_parts, lse_parts):
    """Merge split-K partial states by their log-sum-exps.

    [vllmcpp] MergeAttnStates: lse = log sum_s exp(lse_s), o = sum_s
    exp(lse_s - lse) o_s; a +inf lse is treated as -inf (an empty split).
    When every split is empty the sum is 0/0; that test's reference then
    emits the PREFIX output with lse = -inf, so the result is the first
    part's o (the prefix is part 0) and lse = -inf. (A decode split with no
    keys carries o = 0, so an empty request still yields o = 0.)
    o_parts: [S, G, D]; lse_parts: [S, G].
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse = np.asarray(lse_parts, dtype=np.float64).copy()
    lse[np.isinf(lse)] = -np.inf
    S, G = lse.shape
    o = np.zeros(o_parts.shape[1:])
    out_lse = np.full(G, -np.inf)
    for g in range(G):
        m = lse[:, g].max()
        if not np.isfinite(m):
            o[g] = o_parts[0, g, :]
            continue
        w = np.exp(lse[:, g] - m)
        tot = w.sum()
        o[g] = (w[:, None] * o_parts[:, g, :]).sum(0) / tot
        out_lse[g] = m + math.log(tot)
    return o, out_lse


# ---------------------------------------------------------------------------
# one (request, KV head) unit of the page-level step
# ---------------------------------------------------------------------------
def page_decode_unit(k_head_bits, v_head_bits, L: int, q_group_bits, *, ps: int,
                     topk: int, w_avg: float, w_peak: float, dtype: str,
                     scale: float = 0.0, alpha: float = 1.0):
    """Steps A1 -> A4 for one (request, KV head): page statistics of the L
    cached keys, page scores, top-k with the tail forced, and attention of the
    G query heads over the selected pages' valid tokens -- softmax, or with
    alpha != 1 the alpha-entmax of attention_entmax ([entmax] How it works).

    k_head_bits, v_head_bits: uint16 [L, D]; q_group_bits: uint16 [G, D].
    Returns dict(meta=(mn, mx, me), scores, sel, out [G, D], lse [G]) (with
    entmax: tau [G] in place of lse).
    """
    D = k_head_bits.shape[1]
    sc = scale if scale > 0 else default_scale(D)
    mn, mx, me = head_meta(k_head_bits, L, ps, dtype)
    q = decode_kdt(q_group_bits, dtype)
    scores = score_pages(mn, mx, me, q, w_avg, w_peak)
    sel = select_pages(scores, num_pages(L, ps), topk)
    pos = selected_positions(sel, L, ps)
    k = decode_kdt(k_head_bits[pos], dtype)
    v = decode_kdt(v_head_bits[pos], dtype)
    if alpha != 1.0:
        o, tau, _ = attention_entmax(q, k, v, sc, alpha)
        return {"meta": (mn, mx, me), "scores": scores, "sel": sel, "out": o, "tau": tau}
    o, lse, _ = attention(q, k, v, sc)
    return {"meta": (mn, mx, me), "scores": scores, "sel": sel, "out": o, "lse": lse}


# ---------------------------------------------------------------------------
# A5: token-level H2O accumulate and evict
# ---------------------------------------------------------------------------
def h2o_fold(hh, logits, lse, decay: float) -> np.ndarray:
    """Decayed accumulation of attention probabilities, before storage rounding.

    [vortex] "Token-level variants" points 1 and 3 (accumulate softmax
    probabilities, not logits; out = 1 * attn + decay * old);
    [velox] "How it works" step 2 (scores * decay + attn).
    p_bar_j = (1/G) sum_g exp(z_gj - lse_g); returns decay * hh + p_bar.
    hh: [n]; logits: [G, n]; lse: [G].
    """
    p = np.exp(np.asarray(logits, np.float64) - np.asarray(lse, np.float64)[:, None])
    return decay * np.asarray(hh, np.float64) + p.mean(0)


def h2o_fold_window(hh, logits, n_bos: int, n_eos: int, decay: float) -> np.ndarray:
    """The decayed fold with a reserved window, before storage rounding.

    [vortex] follow-up comment, "Two things I had to fix" and its reference
    step: hh_score is nonzero only between the reserved tokens; the softmax is
    normalised over that window alone and the reserved entries receive
    nothing. Here the reserved entries are the first n_bos and the last n_eos
    of the retained list. hh: [n]; logits: [G, n].
    p_bar_j = (1/G) sum_g exp(z_gj - lse'_g), lse'_g = log sum_{j in window} exp(z_gj).
    """
    z = np.asarray(logits, np.float64)
    n = z.shape[1]
    lo, hi = int(n_bos), n - int(n_eos)
    p = np.zeros_like(z)
    if hi > lo:
        zw = z[:, lo:hi]
        m = zw.max(axis=1, keepdims=True)
        lse_w = m + np.log(np.exp(zw - m).sum(axis=1, keepdims=True))
        p[:, lo:hi] = np.exp(zw - lse_w)
    return decay * np.asarray(hh, np.float64) + p.mean(0)


def h2o_store(hh_exact) -> np.ndarray:
    """[vortex] point 3: hh_score is held in bfloat16 -- one rounding to bf16."""
    return round_to_kdt(hh_exact, "bf16")


def h2o_evict(hh, positions, budget: int, n_sink: int, grace: int):
    """Evict until the retained list holds at most ``budget`` tokens.

    [velox] "Parameters" and "How it works" step 3: the first n_sink entries
    (attention sinks) and the last ``grace`` entries (the newest arrivals, the
    list being kept ascending by position) are protected; the entry with the
    minimum score among the rest is removed, one at a time, the first index
    winning a tie (as mx.argmin does, hence the lowest position).
    Step 4: after the update |R| <= budget.

    hh: scores of the retained entries (in list order); positions: ascending.
    Returns (kept positions, kept scores, evicted positions in eviction order).
    """
    R = [int(p) for p in positions]
    s = [float(x) for x in hh]
    evicted: List[int] = []
    while len(R) > budget:
        lo, hi = n_sink, len(R) - grace
        if hi <= lo:
            raise ValueError("no evictable entry: budget must exceed n_sink + grace")
        j = lo + int(np.argmin(np.asarray(s[lo:hi])))
        evicted.append(R.pop(j))
        s.pop(j)
    return np.asarray(R, dtype=np.int64), np.asarray(s), evicted


def h2o_proxy_token(keys, positions, hh, k_new, pos_new: int, *, decay: float, budget: int,
                    n_sink: int, grace: int, scale: float, store: bool = True):
    """One incoming token of the H2O cache, its own key standing in for the query.

    [velox] "How it works", for every incoming token (prefill and decode), per
    head: 1. the new key attends to every stored key, attn = softmax(K k / sqrt(D))
    (here the given scale); 2. scores = scores * decay + attn; new tokens start
    at 0; 3. above budget the minimum-score entry outside the first n_sink and
    the last grace (the newest) is removed, the first index winning a tie;
    4. at most budget entries remain. With store, scores are held in bf16, the
    fold rounded once as in the decode-side update (a reading: [vortex] point 3).

    keys: float64 [n, D] (list order = ascending positions); returns
    (keys, positions, hh, evicted position or None).
    """
    keys = np.asarray(keys, np.float64).reshape(-1, np.asarray(k_new).shape[-1])
    positions = np.asarray(positions, np.int64)
    hh = np.asarray(hh, np.float64)
    if len(positions):
        z = keys @ np.asarray(k_new, np.float64) * scale
        p = np.exp(z - z.max())
        p /= p.sum()
        hh = decay * hh + p
        if store:
            hh = h2o_store(hh)
    keys = np.vstack([keys, np.asarray(k_new, np.float64)[None, :]])
    positions = np.append(positions, pos_new)
    hh = np.append(hh, 0.0)
    ev = None
    if len(positions) > budget:
        lo, hi = n_sink, len(positions) - grace
        if hi <= lo:
            raise ValueError("no evictable entry: budget must exceed n_sink + grace")
        j = lo + int(np.argmin(hh[lo:hi]))
        ev = int(positions[j])
        keys = np.delete(keys, j, axis=0)
        positions = np.delete(positions, j)
        hh = np.delete(hh, j)
    return keys, positions, hh, ev


def h2o_proxy_prefill(keys_in, pos_in, *, decay: float, budget: int, n_sink: int, grace: int,
                      scale: float, state=None, store: bool = True):
    """h2o_proxy_token over incoming tokens in order (a prefill chunk, or the
    decode tokens), from an optional (keys, positions, hh) state. [velox]
    "How it works" and the below-budget batched absorb of its changelog, which
    it states gives the same scores as this token-by-token loop.
    Returns (keys, positions, hh, evicted positions in order)."""
    D = np.asarray(keys_in).shape[-1]
    keys, pos, hh = state if state is not None else (np.zeros((0, D)), np.zeros(0, np.int64), np.zeros(0))
    evicted = []
    for k, p in zip(np.asarray(keys_in, np.float64), pos_in):
        keys, pos, hh, ev = h2o_proxy_token(keys, pos, hh, k, int(p), decay=decay, budget=budget,
                                            n_sink=n_sink, grace=grace, scale=scale, store=store)
        if ev is not None:
            evicted.append(ev)
    return keys, pos, hh, evicted


def h2o_unit_step(hh_ret, positions, k_head_bits, v_head_bits, q_group_bits, *,
                  dtype: str, decay: float, budget: int, n_sink: int, grace: int,
                  scale: float = 0.0, window_softmax: bool = False):
    """One token-level decode step for one (request, KV head), after the new
    token has been appended to the retained list with hh = 0.

    Attention of the G query heads over the retained tokens (page_size 1, the
    selection is the retained list itself), then the decayed bf16 fold, then
    eviction. hh_ret: bf16 values (float64) of the retained entries in list
    order; positions: their positions (ascending); k/v_head_bits: uint16 [L, D]
    logical keys / values of the request.
    With window_softmax the fold is h2o_fold_window with the protected entries
    (the first n_sink and the last grace) as the reserved ones.
    Returns dict(out, lse, logits, hh_exact, hh_bf16, kept, kept_hh, evicted).
    """
    D = k_head_bits.shape[1]
    sc = scale if scale > 0 else default_scale(D)
    pos = np.asarray(positions, dtype=np.int64)
    q = decode_kdt(q_group_bits, dtype)
    k = decode_kdt(k_head_bits[pos], dtype)
    v = decode_kdt(v_head_bits[pos], dtype)
    o, lse, z = attention(q, k, v, sc)
    hh_exact = (h2o_fold_window(hh_ret, z, n_sink, grace, decay) if window_softmax
                else h2o_fold(hh_ret, z, lse, decay))
    hh_b = h2o_store(hh_exact)
    kept, kept_hh, ev = h2o_evict(hh_b, pos, budget, n_sink, grace)
    return {"out": o, "lse": lse, "logits": z, "hh_exact": hh_exact, "hh_bf16": hh_b,
            "kept": kept, "kept_hh": kept_hh, "evicted": ev}
