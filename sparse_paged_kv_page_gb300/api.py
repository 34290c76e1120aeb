"""Thin torch-tensor binding of the C ABI (include/sparse_attn.h).

Argument marshalling only: every step runs in the native library's CUDA
kernels. Functions keep the C names and argument order; tensors must be CUDA,
contiguous and of the documented dtype; ``stream`` defaults to torch's current
stream. A non-OK status raises :class:`SaError`.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import SaBatch, SaCache

__all__ = ["SaError", "SaCache", "SaBatch", "make_cache", "make_batch", "PagedKVCache",
           "sa_append_kv", "sa_score_pages", "sa_select_topk", "sa_decode_workspace_size",
           "sa_decode_workspace_init", "sa_sparse_decode", "sa_sparse_decode_noalloc",
           "sa_sparse_decode_noalloc_capacity", "sa_h2o_update", "sa_decode_step",
           "sa_select_topk_reserved", "sa_h2o_update_window", "sa_score_pages_qh",
           "sa_sparse_decode_qh", "sa_h2o_prefill", "sa_entmax_workspace_size",
           "alloc_entmax_workspace", "sa_sparse_decode_entmax", "sa_sparse_decode_entmax_qh",
           "sa_gauss_select", "sa_shard_lengths", "sa_shard_selection", "sa_merge_states",
           "batch_view",
           "sa_status_string", "sa_struct_size", "sa_wait_selftest",
           "sa_version", "alloc_decode_workspace"]

_DT = {torch.bfloat16: _lib.SA_BF16, torch.float16: _lib.SA_FP16}


class SaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {sa_status_string(status)} ({status})")


def _check(fn, st):
    if st != 0:
        raise SaError(fn, st)


def _p(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_cache(k: torch.Tensor, v: torch.Tensor, meta: Optional[torch.Tensor],
               kstd: Optional[torch.Tensor] = None) -> SaCache:
    """Struct view of pools [num_blocks, H_kv, page_size, D], meta [num_blocks, H_kv, 3, D]
    and (optional) kstd [num_blocks, H_kv, D]."""
    if k.dtype not in _DT or v.dtype != k.dtype or k.shape != v.shape or k.dim() != 4:
        raise ValueError("k, v must be bf16/fp16 [num_blocks, H_kv, page_size, D] of equal shape")
    nb, hkv, ps, d = k.shape
    if meta is not None and (meta.dtype != k.dtype or tuple(meta.shape) != (nb, hkv, 3, d)):
        raise ValueError("meta must be [num_blocks, H_kv, 3, D] in the pool dtype")
    if kstd is not None and (kstd.dtype != k.dtype or tuple(kstd.shape) != (nb, hkv, d)):
        raise ValueError("kstd must be [num_blocks, H_kv, D] in the pool dtype")
    c = SaCache(_p(k, name="k"), _p(v, name="v"), _p(meta, name="meta"), _DT[k.dtype], nb, hkv,
                ps, d, _p(kstd, name="kstd"))
    c._keep = (k, v, meta, kstd)
    return c


def make_batch(block_table: torch.Tensor, seq_lens: torch.Tensor) -> SaBatch:
    """Struct view of block_table [B, bt_stride] int32 and seq_lens [B] int32."""
    if block_table.dim() != 2 or seq_lens.dim() != 1 or seq_lens.shape[0] != block_table.shape[0]:
        raise ValueError("block_table [B, stride] and seq_lens [B] expected")
    b = SaBatch(_p(block_table, torch.int32, "block_table"), _p(seq_lens, torch.int32, "seq_lens"),
                block_table.shape[0], block_table.shape[1])
    b._keep = (block_table, seq_lens)
    return b


class PagedKVCache:
    """Device buffers of one paged cache (PyTorch allocates; kernels do the work)."""

    def __init__(self, num_blocks, num_kv_heads, page_size, head_dim, dtype=torch.bfloat16,
                 device="cuda", with_meta=True, with_hh=False, with_std=False):
        shape = (num_blocks, num_kv_heads, page_size, head_dim)
        self.k = torch.empty(shape, dtype=dtype, device=device)
        self.v = torch.empty(shape, dtype=dtype, device=device)
        self.meta = (torch.empty((num_blocks, num_kv_heads, 3, head_dim), dtype=dtype, device=device)
                     if with_meta else None)
        self.hh = (torch.zeros((num_blocks * page_size, num_kv_heads), dtype=torch.bfloat16,
                               device=device) if with_hh else None)
        self.kstd = (torch.empty((num_blocks, num_kv_heads, head_dim), dtype=dtype, device=device)
                     if with_std else None)
        self.struct = make_cache(self.k, self.v, self.meta, self.kstd)


def sa_status_string(status: int) -> str:
    return _lib.load().sa_status_string(int(status)).decode()


def sa_struct_size(which: int) -> int:
    """sizeof(sa_cache) (0) or sizeof(sa_batch) (1) as the library was built."""
    return int(_lib.load().sa_struct_size(int(which)))


def sa_version() -> str:
    return _lib.load().sa_version().decode()


def sa_append_kv(cache: SaCache, batch: SaBatch, k_new, v_new, new_cu, max_new_per_req: int,
                 hh=None, ret_pos=None, ret_cnt=None, ret_cap: int = 0, dev_status=None,
                 stream=None):
    lib = _lib.load()
    _check("sa_append_kv", lib.sa_append_kv(
        ctypes.byref(cache), ctypes.byref(batch), _p(k_new, name="k_new"), _p(v_new, name="v_new"),
        _p(new_cu, torch.int32, "new_cu"), int(max_new_per_req),
        _p(hh, torch.bfloat16, "hh"), _p(ret_pos, torch.int32, "ret_pos"),
        _p(ret_cnt, torch.int32, "ret_cnt"), int(ret_cap),
        _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_score_pages(cache: SaCache, batch: SaBatch, q, num_q_heads: int, w_avg: float,
                   w_peak: float, scores, max_pages: int, dev_status=None, stream=None):
    lib = _lib.load()
    _check("sa_score_pages", lib.sa_score_pages(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads),
        float(w_avg), float(w_peak), _p(scores, torch.float32, "scores"), int(max_pages),
        _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_score_pages_qh(cache: SaCache, batch: SaBatch, q, num_q_heads: int, w_avg: float,
                      w_peak: float, scores, max_pages: int, dev_status=None, stream=None):
    """One score row per query head: scores [B, H_q, max_pages]."""
    lib = _lib.load()
    _check("sa_score_pages_qh", lib.sa_score_pages_qh(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads),
        float(w_avg), float(w_peak), _p(scores, torch.float32, "scores"), int(max_pages),
        _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_sparse_decode_qh(cache: SaCache, batch: SaBatch, q, num_q_heads: int, sel_idx, sel_cnt,
                        sel_stride: int, scale: float, out, lse=None, workspace=None,
                        dev_status=None, stream=None):
    """Attention with a selection per query head: sel_idx [B, H_q, sel_stride]."""
    lib = _lib.load()
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("sa_sparse_decode_qh", lib.sa_sparse_decode_qh(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads),
        _p(sel_idx, torch.int32, "sel_idx"), _p(sel_cnt, torch.int32, "sel_cnt"), int(sel_stride),
        float(scale), _p(out, name="out"), _p(lse, torch.float32, "lse"),
        _p(workspace, name="workspace"), wbytes, _p(dev_status, torch.int32, "dev_status"),
        _s(stream)))


def sa_select_topk(scores, max_pages: int, batch: SaBatch, page_size: int, num_kv_heads: int,
                   topk: int, sel_idx, sel_cnt, dev_status=None, stream=None):
    lib = _lib.load()
    _check("sa_select_topk", lib.sa_select_topk(
        _p(scores, torch.float32, "scores"), int(max_pages), ctypes.byref(batch), int(page_size),
        int(num_kv_heads), int(topk), _p(sel_idx, torch.int32, "sel_idx"),
        _p(sel_cnt, torch.int32, "sel_cnt"), _p(dev_status, torch.int32, "dev_status"),
        _s(stream)))


def sa_select_topk_reserved(scores, max_pages: int, batch: SaBatch, page_size: int,
                            num_kv_heads: int, topk: int, n_bos: int, n_eos: int, sel_idx,
                            sel_cnt, dev_status=None, stream=None):
    lib = _lib.load()
    _check("sa_select_topk_reserved", lib.sa_select_topk_reserved(
        _p(scores, torch.float32, "scores"), int(max_pages), ctypes.byref(batch), int(page_size),
        int(num_kv_heads), int(topk), int(n_bos), int(n_eos), _p(sel_idx, torch.int32, "sel_idx"),
        _p(sel_cnt, torch.int32, "sel_cnt"), _p(dev_status, torch.int32, "dev_status"),
        _s(stream)))


def sa_decode_workspace_size(batch: int, num_kv_heads: int, num_q_heads: int, head_dim: int,
                             page_size: int, sel_stride: int) -> int:
    return int(_lib.load().sa_decode_workspace_size(batch, num_kv_heads, num_q_heads, head_dim,
                                                    page_size, sel_stride))


def sa_decode_workspace_init(workspace, stream=None):
    _check("sa_decode_workspace_init", _lib.load().sa_decode_workspace_init(
        _p(workspace, name="workspace"), workspace.numel() * workspace.element_size(), _s(stream)))


def alloc_decode_workspace(batch, num_kv_heads, num_q_heads, head_dim, page_size, sel_stride,
                           device="cuda"):
    """A zero-filled workspace tensor of the size sa_sparse_decode needs."""
    n = max(256, sa_decode_workspace_size(batch, num_kv_heads, num_q_heads, head_dim, page_size,
                                          sel_stride))
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sa_sparse_decode(cache: SaCache, batch: SaBatch, q, num_q_heads: int, sel_idx, sel_cnt,
                     sel_stride: int, scale: float, out, lse=None, logits=None,
                     logits_stride: int = 0, workspace=None, dev_status=None, stream=None):
    lib = _lib.load()
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("sa_sparse_decode", lib.sa_sparse_decode(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads),
        _p(sel_idx, torch.int32, "sel_idx"), _p(sel_cnt, torch.int32, "sel_cnt"), int(sel_stride),
        float(scale), _p(out, name="out"), _p(lse, torch.float32, "lse"),
        _p(logits, torch.float32, "logits"), int(logits_stride), _p(workspace, name="workspace"),
        wbytes, _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_entmax_workspace_size(batch: int, num_kv_heads: int, num_q_heads: int, head_dim: int,
                             page_size: int, sel_stride: int) -> int:
    return int(_lib.load().sa_entmax_workspace_size(int(batch), int(num_kv_heads), int(num_q_heads),
                                                    int(head_dim), int(page_size), int(sel_stride)))


def alloc_entmax_workspace(batch, num_kv_heads, num_q_heads, head_dim, page_size, sel_stride,
                           device="cuda"):
    """A zero-filled workspace tensor of the size sa_sparse_decode_entmax needs."""
    n = max(256, sa_entmax_workspace_size(batch, num_kv_heads, num_q_heads, head_dim, page_size,
                                          sel_stride))
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sa_sparse_decode_entmax(cache: SaCache, batch: SaBatch, q, num_q_heads: int, sel_idx, sel_cnt,
                            sel_stride: int, alpha: float, scale: float, out, tau=None, logits=None,
                            logits_stride: int = 0, workspace=None, dev_status=None, stream=None):
    """Attention over the selection with alpha-entmax (1 < alpha <= 2) in place of the softmax."""
    lib = _lib.load()
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("sa_sparse_decode_entmax", lib.sa_sparse_decode_entmax(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads),
        _p(sel_idx, torch.int32, "sel_idx"), _p(sel_cnt, torch.int32, "sel_cnt"), int(sel_stride),
        float(alpha), float(scale), _p(out, name="out"), _p(tau, torch.float32, "tau"),
        _p(logits, torch.float32, "logits"), int(logits_stride), _p(workspace, name="workspace"),
        wbytes, _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_sparse_decode_entmax_qh(cache: SaCache, batch: SaBatch, q, num_q_heads: int, sel_idx,
                               sel_cnt, sel_stride: int, alpha: float, scale: float, out, tau=None,
                               logits=None, logits_stride: int = 0, workspace=None,
                               dev_status=None, stream=None):
    """sa_sparse_decode_entmax with a selection per query head: sel_idx [B, H_q, sel_stride]
    (workspace: alloc_entmax_workspace(B, H_q, H_q, ...))."""
    lib = _lib.load()
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("sa_sparse_decode_entmax_qh", lib.sa_sparse_decode_entmax_qh(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads),
        _p(sel_idx, torch.int32, "sel_idx"), _p(sel_cnt, torch.int32, "sel_cnt"), int(sel_stride),
        float(alpha), float(scale), _p(out, name="out"), _p(tau, torch.float32, "tau"),
        _p(logits, torch.float32, "logits"), int(logits_stride), _p(workspace, name="workspace"),
        wbytes, _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_gauss_select(cache: SaCache, batch: SaBatch, q, num_q_heads: int, alpha: float,
                    scale: float, moments, max_pages: int, sel_idx, sel_cnt, sel_stride: int,
                    tau_hat=None, dev_status=None, stream=None):
    """Gaussian-aware selection per query head: moments float32 [B, H_q, max_pages, 2]
    (scratch), sel_idx [B, H_q, sel_stride], sel_cnt [B, H_q], tau_hat [B, H_q]."""
    lib = _lib.load()
    _check("sa_gauss_select", lib.sa_gauss_select(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads), float(alpha),
        float(scale), _p(moments, torch.float32, "moments"), int(max_pages),
        _p(sel_idx, torch.int32, "sel_idx"), _p(sel_cnt, torch.int32, "sel_cnt"), int(sel_stride),
        _p(tau_hat, torch.float32, "tau_hat"), _p(dev_status, torch.int32, "dev_status"),
        _s(stream)))


def sa_shard_lengths(seq_lens, batch: int, page_size: int, page_lo: int, page_hi: int, shard_lens,
                     stream=None):
    _check("sa_shard_lengths", _lib.load().sa_shard_lengths(
        _p(seq_lens, torch.int32, "seq_lens"), int(batch), int(page_size), int(page_lo), int(page_hi),
        _p(shard_lens, torch.int32, "shard_lens"), _s(stream)))


def sa_shard_selection(sel_idx, sel_cnt, sel_stride: int, num_units: int, page_lo: int, page_hi: int,
                       shard_idx, shard_cnt, shard_stride: int, dev_status=None, stream=None):
    _check("sa_shard_selection", _lib.load().sa_shard_selection(
        _p(sel_idx, torch.int32, "sel_idx"), _p(sel_cnt, torch.int32, "sel_cnt"), int(sel_stride),
        int(num_units), int(page_lo), int(page_hi), _p(shard_idx, torch.int32, "shard_idx"),
        _p(shard_cnt, torch.int32, "shard_cnt"), int(shard_stride),
        _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_merge_states(o_parts, lse_parts, num_shards: int, rows: int, head_dim: int, out, lse=None,
                    stream=None):
    if o_parts.dtype not in _DT or out.dtype != o_parts.dtype:
        raise ValueError("o_parts and out must share a bf16/fp16 dtype")
    _check("sa_merge_states", _lib.load().sa_merge_states(
        _p(o_parts, name="o_parts"), _p(lse_parts, torch.float32, "lse_parts"), int(num_shards),
        int(rows), int(head_dim), _DT[o_parts.dtype], _p(out, name="out"),
        _p(lse, torch.float32, "lse"), _s(stream)))


def sa_wait_selftest(arrivals: int, limit_ns: int, dev_status, result, stream=None):
    """The library's bounded in-kernel wait on an mbarrier given `arrivals` of
    its 2 expected arrivals (fewer: it runs out after limit_ns, sets
    SA_DEV_TIMEOUT and writes result = 0)."""
    _check("sa_wait_selftest", _lib.load().sa_wait_selftest(
        int(arrivals), int(limit_ns), _p(dev_status, torch.int32, "dev_status"),
        _p(result, torch.int32, "result"), _s(stream)))


def batch_view(block_table: torch.Tensor, seq_lens: torch.Tensor, page_lo: int) -> SaBatch:
    """Struct view of pages [page_lo, ...) of every row of block_table [B, bt_stride]
    (the same row stride), with the shard's own lengths seq_lens [B]."""
    if block_table.dtype != torch.int32 or not block_table.is_contiguous() or block_table.dim() != 2:
        raise ValueError("block_table must be contiguous int32 [B, bt_stride]")
    if not 0 <= page_lo < block_table.shape[1]:
        raise ValueError("page_lo outside the table")
    b = SaBatch(ctypes.c_void_p(block_table.data_ptr() + 4 * int(page_lo)),
                _p(seq_lens, torch.int32, "seq_lens"), int(block_table.shape[0]),
                int(block_table.shape[1]))
    b._keep = (block_table, seq_lens)
    return b


def sa_sparse_decode_noalloc(cache: SaCache, batch: SaBatch, q, num_q_heads: int, sel_idx,
                             sel_cnt, sel_stride: int, scale: float, out, lse=None, logits=None,
                             logits_stride: int = 0, dev_status=None, stream=None):
    """sa_sparse_decode with the library's fixed scratch instead of a workspace
    (for callers that cannot allocate; calls must not overlap on the GPU)."""
    lib = _lib.load()
    _check("sa_sparse_decode_noalloc", lib.sa_sparse_decode_noalloc(
        ctypes.byref(cache), ctypes.byref(batch), _p(q, name="q"), int(num_q_heads),
        _p(sel_idx, torch.int32, "sel_idx"), _p(sel_cnt, torch.int32, "sel_cnt"), int(sel_stride),
        float(scale), _p(out, name="out"), _p(lse, torch.float32, "lse"),
        _p(logits, torch.float32, "logits"), int(logits_stride),
        _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_sparse_decode_noalloc_capacity() -> int:
    return int(_lib.load().sa_sparse_decode_noalloc_capacity())


def _h2o(name, batch: SaBatch, num_kv_heads: int, num_q_heads: int, logits, logits_stride: int,
         lse, hh, num_slots: int, ret_pos, ret_cnt, ret_cap: int, budget: int, n_sink: int,
         grace: int, decay: float, evicted=None, evicted_cnt=None, dev_status=None, stream=None):
    lib = _lib.load()
    _check(name, getattr(lib, name)(
        ctypes.byref(batch), int(num_kv_heads), int(num_q_heads),
        _p(logits, torch.float32, "logits"), int(logits_stride), _p(lse, torch.float32, "lse"),
        _p(hh, torch.bfloat16, "hh"), int(num_slots), _p(ret_pos, torch.int32, "ret_pos"),
        _p(ret_cnt, torch.int32, "ret_cnt"), int(ret_cap), int(budget), int(n_sink), int(grace),
        float(decay), _p(evicted, torch.int32, "evicted"),
        _p(evicted_cnt, torch.int32, "evicted_cnt"), _p(dev_status, torch.int32, "dev_status"),
        _s(stream)))


def sa_h2o_update(batch: SaBatch, num_kv_heads: int, num_q_heads: int, logits,
                  logits_stride: int, lse, hh, num_slots: int, ret_pos, ret_cnt, ret_cap: int,
                  budget: int, n_sink: int, grace: int, decay: float, evicted=None,
                  evicted_cnt=None, dev_status=None, stream=None):
    _h2o("sa_h2o_update", batch, num_kv_heads, num_q_heads, logits, logits_stride, lse, hh,
         num_slots, ret_pos, ret_cnt, ret_cap, budget, n_sink, grace, decay, evicted, evicted_cnt,
         dev_status, stream)


def sa_h2o_update_window(batch: SaBatch, num_kv_heads: int, num_q_heads: int, logits,
                         logits_stride: int, lse, hh, num_slots: int, ret_pos, ret_cnt,
                         ret_cap: int, budget: int, n_sink: int, grace: int, decay: float,
                         evicted=None, evicted_cnt=None, dev_status=None, stream=None):
    """sa_h2o_update with the softmax normalised over the unprotected entries."""
    _h2o("sa_h2o_update_window", batch, num_kv_heads, num_q_heads, logits, logits_stride, lse,
         hh, num_slots, ret_pos, ret_cnt, ret_cap, budget, n_sink, grace, decay, evicted,
         evicted_cnt, dev_status, stream)


def sa_decode_step(cache: SaCache, batch: SaBatch, k_new, v_new, new_cu, max_new_per_req: int,
                   q, num_q_heads: int, w_avg: float, w_peak: float, scores, max_pages: int,
                   topk: int, sel_idx, sel_cnt, scale: float, out, lse=None, workspace=None,
                   dev_status=None, stream=None, n_bos: int = 0, n_eos: int = 1):
    """Append (k_new may be None), score, select (reserved pages n_bos / n_eos)
    and decode in one chained call."""
    lib = _lib.load()
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("sa_decode_step", lib.sa_decode_step(
        ctypes.byref(cache), ctypes.byref(batch), _p(k_new, name="k_new"), _p(v_new, name="v_new"),
        _p(new_cu, torch.int32, "new_cu"), int(max_new_per_req), _p(q, name="q"),
        int(num_q_heads), float(w_avg), float(w_peak), _p(scores, torch.float32, "scores"),
        int(max_pages), int(topk), int(n_bos), int(n_eos), _p(sel_idx, torch.int32, "sel_idx"),
        _p(sel_cnt, torch.int32, "sel_cnt"), float(scale), _p(out, name="out"),
        _p(lse, torch.float32, "lse"), _p(workspace, name="workspace"), wbytes,
        _p(dev_status, torch.int32, "dev_status"), _s(stream)))


def sa_h2o_prefill(cache: SaCache, batch: SaBatch, new_cu, hh, num_slots: int, ret_pos, ret_cnt,
                   ret_cap: int, budget: int, n_sink: int, grace: int, decay: float,
                   scale: float = 0.0, evicted=None, evicted_cnt=None, dev_status=None,
                   stream=None):
    """H2O absorb / eviction of the tokens just appended, each new key as the query."""
    lib = _lib.load()
    ev_cap = 0 if evicted is None else evicted.shape[-1]
    _check("sa_h2o_prefill", lib.sa_h2o_prefill(
        ctypes.byref(cache), ctypes.byref(batch), _p(new_cu, torch.int32, "new_cu"),
        _p(hh, torch.bfloat16, "hh"), int(num_slots), _p(ret_pos, torch.int32, "ret_pos"),
        _p(ret_cnt, torch.int32, "ret_cnt"), int(ret_cap), int(budget), int(n_sink), int(grace),
        float(decay), float(scale), _p(evicted, torch.int32, "evicted"),
        _p(evicted_cnt, torch.int32, "evicted_cnt"), int(ev_cap),
        _p(dev_status, torch.int32, "dev_status"), _s(stream)))
