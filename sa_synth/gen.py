"""Seeded synthetic inputs for the paged sparse-decode step.

Both sides of every parity check (the CUDA path and the CPU oracle) draw their
inputs from here, and only from here. The module draws random numbers
(numpy PCG64, one sub-stream per (kind, request, chunk) so results do not
depend on thread count), shapes them into the workload's value structure,
builds block tables, and encodes values as bf16/fp16 bit patterns. The
float32 -> bf16/fp16 encoding is torch's round-to-nearest-even cast. It holds
none of the method's arithmetic (no statistics, scores, selection, softmax or
accumulation).

Value recipes (``Config.structure``):

* ``iid``                Q, K, V ~ N(0, 1).
* ``page_unit_offset``   keys of page p get ``+0.5 * u_p`` (u_p a random unit
                         vector per page) so pages differ.
* ``page_normal_offset`` keys of page p, KV head h get ``+a_p * u_h`` with
                         a_p ~ N(0, 0.5^2) and u_h one unit vector per KV head.
* ``hot_pages_corr``     5% of pages (Bernoulli per request page) get keys
                         ``+1.0 * d_bh``; d_bh is a unit direction with
                         cos(d_bh, u_bh) = 0.7 where u_bh is the normalised
                         sum of the step's G queries of that KV head.
* ``hot_pages_qdir``     fixed unit u_h per KV head; queries are
                         ``N(0,1) + 1.0 * u_h``; 1% of pages get keys
                         ``+1.5 * u_h``.
* ``heavy_hitters``      token-level: keys carry a stable per-token affinity
                         ``a_j * u`` (a_j ~ N(0, 2^2), u one shared unit vector)
                         and queries lean towards u (``0.3 * N(0,1) + u``), so the
                         same tokens attract attention step after step.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Tuple

import numpy as np

from .configs import Config

_CHUNK = 1 << 22            # values per generator chunk
_THREADS = 16


# --------------------------------------------------------------------------
# encoding
# --------------------------------------------------------------------------
def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> uint16 bit patterns of bf16/fp16 (round to nearest even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return t.to(tdt).view(torch.int16).numpy().view(np.uint16)


def _normal(shape, key, scale: float = 1.0) -> np.ndarray:
    """float32 N(0, scale^2) of the given shape, chunk-seeded by ``key``."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nch = (n + _CHUNK - 1) // _CHUNK

    def work(i):
        rng = np.random.default_rng(list(key) + [i])
        s = slice(i * _CHUNK, min(n, (i + 1) * _CHUNK))
        rng.standard_normal(out=out[s], dtype=np.float32)

    if nch <= 1:
        for i in range(nch):
            work(i)
    else:
        with ThreadPoolExecutor(min(_THREADS, nch)) as ex:
            list(ex.map(work, range(nch)))
    if scale != 1.0:
        out *= np.float32(scale)
    return out.reshape(shape)


def _unit(rng, *shape) -> np.ndarray:
    v = rng.standard_normal(shape)
    return v / np.linalg.norm(v, axis=-1, keepdims=True)


# --------------------------------------------------------------------------
# block tables
# --------------------------------------------------------------------------
def reverse_interleaved(B: int, max_pages: int, num_blocks: int) -> np.ndarray:
    """Request b's logical page p -> physical block num_blocks-1-(p*B+b).

    The adversarial table of the vllm.cpp chunked-context test
    ("test_ops_mla_chunked_context.cpp", GatherMlaCache case): nothing is
    contiguous or ascending.
    """
    p = np.arange(max_pages, dtype=np.int64)[None, :]
    b = np.arange(B, dtype=np.int64)[:, None]
    bt = num_blocks - 1 - (p * B + b)
    if bt.min() < 0:
        raise ValueError("reverse-interleaved table needs num_blocks >= B * max_pages")
    return bt.astype(np.int32)


def contiguous_table(B: int, max_pages: int) -> np.ndarray:
    return (np.arange(B * max_pages, dtype=np.int64).reshape(B, max_pages)).astype(np.int32)


def shuffled_table(B: int, max_pages: int, pages_needed, num_blocks: int, rng) -> np.ndarray:
    """A random permutation of the physical blocks handed out in request order."""
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        n = int(pages_needed[b])
        bt[b, :n] = perm[o:o + n]
        o += n
    return bt


# --------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------
class Workload:
    """All inputs of one workload, as bit patterns and int32 tables.

    Attributes
    ----------
    prefill_lens : int32 [B]          tokens per request before the first decode step
    pre_cu       : int32 [B+1]        row offsets of each request in k_pre / v_pre
    k_pre, v_pre : uint16 [T, H_kv, D] prefill keys / values, requests concatenated
    block_table  : int32 [B, max_pages]
    num_blocks   : physical blocks (token slots when ps == 1)
    max_pages    : table stride (capacity in pages per request)
    q(t), kv_new(t): per-decode-step queries [B, H_q, D] and new keys/values [B, H_kv, D]
    """

    def __init__(self, cfg: Config, extra_steps: int = 0):
        self.cfg = cfg
        c = cfg
        seed = c.rng_seed
        self._seed = seed
        srng = np.random.default_rng([seed, 0])
        B = c.B
        if c.prefill is not None:
            lens = np.asarray(c.prefill, dtype=np.int64)
            assert lens.shape == (B,)
        else:
            lo, hi = c.len_range
            lens = srng.integers(lo, hi + 1, size=B)
        self.prefill_lens = lens.astype(np.int32)
        steps = max(c.decode_steps, 0) + extra_steps
        self.total_steps = steps
        final = lens + steps
        ps = c.ps
        pages_needed = (final + ps - 1) // ps
        self.max_pages = int(max(1, pages_needed.max()))
        # structure parameters (drawn before tables so they do not depend on table type)
        self._struct = self._draw_structure(srng)
        nb = c.num_blocks
        if c.table == "reverse":
            need = B * self.max_pages
            nb = max(nb or 0, need)
            self.block_table = reverse_interleaved(B, self.max_pages, nb)
        elif c.table == "contiguous":
            need = B * self.max_pages
            nb = max(nb or 0, need)
            self.block_table = contiguous_table(B, self.max_pages)
        elif c.table == "shuffle":
            need = int(pages_needed.sum())
            nb = max(nb or 0, need)
            self.block_table = shuffled_table(B, self.max_pages, pages_needed, nb,
                                              np.random.default_rng([seed, 6]))
        else:
            raise ValueError(c.table)
        self.num_blocks = int(nb)
        self.pre_cu = np.zeros(B + 1, dtype=np.int32)
        self.pre_cu[1:] = np.cumsum(lens)
        self.k_pre, self.v_pre = self._prefill()

    # ---- structure -------------------------------------------------------
    def _draw_structure(self, rng):
        c = self.cfg
        s = {}
        ps, B = c.ps, c.B
        cap_pages = int(((self.prefill_lens.max() + self.total_steps + 4096) + ps - 1) // ps)
        if c.structure == "page_unit_offset":
            s["u_page"] = _unit(rng, B, cap_pages, c.D).astype(np.float32)
        elif c.structure == "page_normal_offset":
            s["a_page"] = (rng.standard_normal((B, cap_pages)) * 0.5).astype(np.float32)
            s["u_head"] = _unit(rng, c.H_kv, c.D).astype(np.float32)
        elif c.structure == "hot_pages_corr":
            s["hot"] = rng.random((B, cap_pages)) < 0.05
            q0 = self._q_float(0)                       # [B, H_q, D]
            qg = q0.reshape(B, c.H_kv, c.G, c.D).sum(2).astype(np.float64)
            u = qg / np.linalg.norm(qg, axis=-1, keepdims=True)
            w = rng.standard_normal(u.shape)
            w -= (w * u).sum(-1, keepdims=True) * u
            w /= np.linalg.norm(w, axis=-1, keepdims=True)
            d = 0.7 * u + math.sqrt(0.51) * w
            s["dir"] = d.astype(np.float32)             # [B, H_kv, D]
        elif c.structure == "hot_pages_qdir":
            s["hot"] = rng.random((B, cap_pages)) < 0.01
            s["u_head"] = _unit(rng, c.H_kv, c.D).astype(np.float32)
        elif c.structure == "heavy_hitters":
            s["u"] = _unit(rng, c.D).astype(np.float32)
            s["aff"] = (rng.standard_normal((B, cap_pages * ps)) * 2.0).astype(np.float32)
        elif c.structure == "iid":
            pass
        else:
            raise ValueError(c.structure)
        s["cap_pages"] = cap_pages
        return s

    def _key_offset(self, b: int, pos: np.ndarray) -> Optional[np.ndarray]:
        """Structured offset added to keys at positions ``pos`` of request b: [n, H_kv, D]."""
        c, s = self.cfg, self._struct
        page = pos // c.ps
        if c.structure == "page_unit_offset":
            off = 0.5 * s["u_page"][b, page]                          # [n, D]
            return np.broadcast_to(off[:, None, :], (len(pos), c.H_kv, c.D))
        if c.structure == "page_normal_offset":
            return s["a_page"][b, page][:, None, None] * s["u_head"][None, :, :]
        if c.structure == "hot_pages_corr":
            hot = s["hot"][b, page].astype(np.float32)
            return hot[:, None, None] * 1.0 * s["dir"][b][None, :, :]
        if c.structure == "hot_pages_qdir":
            hot = s["hot"][b, page].astype(np.float32)
            return hot[:, None, None] * 1.5 * s["u_head"][None, :, :]
        if c.structure == "heavy_hitters":
            a = s["aff"][b, pos]
            return np.broadcast_to((a[:, None] * s["u"][None, :])[:, None, :],
                                   (len(pos), c.H_kv, c.D))
        return None

    def _prefill(self):
        c = self.cfg
        Ks, Vs = [], []
        for b in range(c.B):
            L = int(self.prefill_lens[b])
            k = _normal((L, c.H_kv, c.D), [self._seed, 2, b])
            v = _normal((L, c.H_kv, c.D), [self._seed, 3, b])
            off = self._key_offset(b, np.arange(L))
            if off is not None:
                if c.structure in ("hot_pages_corr", "hot_pages_qdir"):
                    page = np.arange(L) // c.ps
                    hot = self._struct["hot"][b, page]
                    k[hot] += off[hot]
                else:
                    k += off
            Ks.append(encode(k, c.dtype))
            Vs.append(encode(v, c.dtype))
        return np.concatenate(Ks, 0), np.concatenate(Vs, 0)

    # ---- per-step inputs -------------------------------------------------
    def _q_float(self, t: int) -> np.ndarray:
        c = self.cfg
        rng = np.random.default_rng([self._seed, 1, t])
        q = rng.standard_normal((c.B, c.H_q, c.D), dtype=np.float32)
        if c.structure == "hot_pages_qdir":
            u = self._struct["u_head"]                                 # [H_kv, D]
            q += np.repeat(u, c.G, axis=0)[None, :, :]
        elif c.structure == "heavy_hitters":
            q = 0.3 * q + self._struct["u"][None, None, :]
        return q

    def q(self, t: int) -> np.ndarray:
        """uint16 [B, H_q, D] query of decode step t (t = 0 is the first step)."""
        return encode(self._q_float(t), self.cfg.dtype)

    def kv_new(self, t: int) -> Tuple[np.ndarray, np.ndarray]:
        """uint16 [B, H_kv, D] key and value appended at decode step t."""
        cache = self.__dict__.setdefault("_kv_cache", {})
        if t not in cache:
            cache[t] = self._kv_new(t)
        return cache[t]

    def _kv_new(self, t: int) -> Tuple[np.ndarray, np.ndarray]:
        c = self.cfg
        k = np.random.default_rng([self._seed, 4, t]).standard_normal((c.B, c.H_kv, c.D), dtype=np.float32)
        v = np.random.default_rng([self._seed, 5, t]).standard_normal((c.B, c.H_kv, c.D), dtype=np.float32)
        for b in range(c.B):
            pos = np.array([int(self.prefill_lens[b]) + t])
            off = self._key_offset(b, pos)
            if off is not None:
                k[b] += off[0]
        return encode(k, c.dtype), encode(v, c.dtype)

    def seq_len(self, b: int, steps_done: int) -> int:
        """Length of request b after ``steps_done`` decode-step appends."""
        return int(self.prefill_lens[b]) + steps_done

    def k_seq(self, b: int, steps_done: int = 0, head: Optional[int] = None) -> np.ndarray:
        """Logical keys of request b (prefill then appended), uint16 [L, H_kv, D]
        (or [L, D] of one KV head when ``head`` is given)."""
        return self._seq(b, steps_done, 0, head)

    def v_seq(self, b: int, steps_done: int = 0, head: Optional[int] = None) -> np.ndarray:
        return self._seq(b, steps_done, 1, head)

    def _seq(self, b, steps_done, which, head=None):
        src = self.k_pre if which == 0 else self.v_pre
        rows = src[self.pre_cu[b]:self.pre_cu[b + 1]]
        if head is not None:
            rows = rows[:, head]
        if steps_done == 0:
            return rows
        if head is None:
            new = np.stack([self.kv_new(t)[which][b] for t in range(steps_done)], 0)
        else:
            new = np.stack([self.kv_new(t)[which][b, head] for t in range(steps_done)], 0)
        return np.concatenate([rows, new], 0)


def make_workload(cfg: Config, extra_steps: int = 0) -> Workload:
    return Workload(cfg, extra_steps=extra_steps)


def fill_stale(t, mode: str, seed: int):
    """Fill a device tensor with stale contents: ``normal3`` = N(0, 3^2), ``nan`` = NaN."""
    import torch
    if mode == "nan":
        t.fill_(float("nan"))
    elif mode == "normal3":
        g = torch.Generator(device=t.device).manual_seed(seed)
        tmp = torch.empty(t.shape, dtype=torch.float32, device=t.device)
        tmp.normal_(0.0, 3.0, generator=g)
        t.copy_(tmp)
    elif mode == "zero":
        t.zero_()
    else:
        raise ValueError(mode)
    return t
