"""Decode-step driver: device buffers plus the per-step chain of C-ABI calls.

Page level (page_size > 1):  append -> score -> select -> sparse decode, one
                             ``sa_decode_step`` call (the append of a single
                             token runs beside the scorer; the tail page's
                             score entry is then unspecified).
Token level (page_size 1):   append (+ retained list) -> sparse decode over
                             the retained tokens (logits + lse) -> H2O update.
alpha-entmax (1 < alpha <= 2, page level): append -> score -> select ->
                             ``sa_sparse_decode_entmax`` (the selection
                             normalised by alpha-entmax instead of softmax).
Gaussian-aware (alpha 1.5 or 2, page level): append (k_mean, k_std) ->
                             ``sa_gauss_select`` (per query head, adaptive
                             count) -> ``sa_sparse_decode_entmax_qh``.

PyTorch only allocates the buffers and supplies the stream; every step runs in
the native kernels. ``capture()`` records one step into a CUDA graph whose
replay needs only the persistent input buffers ``q_buf`` / ``k_buf`` /
``v_buf`` to be refreshed.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from .api import (PagedKVCache, alloc_decode_workspace, alloc_entmax_workspace, make_batch,
                  sa_append_kv, sa_decode_step, sa_h2o_prefill, sa_h2o_update,
                  sa_h2o_update_window, sa_score_pages, sa_score_pages_qh,
                  sa_select_topk_reserved, sa_sparse_decode, sa_sparse_decode_entmax,
                  sa_sparse_decode_entmax_qh, sa_gauss_select, sa_sparse_decode_qh)


class SparseDecoder:
    def __init__(self, *, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 page_size: int, num_blocks: int, bt_stride: int, dtype=torch.bfloat16,
                 topk: int = 0, w_avg: float = 1.0, w_peak: float = 0.25, scale: float = 0.0,
                 budget: int = 0, n_sink: int = 0, grace: int = 0, decay: float = 1.0,
                 ret_cap: int = 0, n_bos: int = 0, n_eos: int = 1, window_softmax: bool = False,
                 per_query_head: bool = False, proxy_prefill: bool = False, alpha: float = 1.0,
                 gaussian: bool = False, device="cuda"):
        self.B, self.H_q, self.H_kv, self.D = batch, num_q_heads, num_kv_heads, head_dim
        self.ps, self.dtype, self.device = page_size, dtype, torch.device(device)
        self.token_level = page_size == 1 and ret_cap > 0
        self.topk, self.w_avg, self.w_peak, self.scale = topk, w_avg, w_peak, scale
        self.budget, self.n_sink, self.grace, self.decay = budget, n_sink, grace, decay
        self.n_bos, self.n_eos, self.window_softmax = n_bos, n_eos, window_softmax
        # per-query-head selection: score, select and attend one row per query head
        self.qh = per_query_head and not self.token_level
        # token level: trim a prefill H2O-style as it arrives (each key as its own query)
        self.proxy_prefill = proxy_prefill and self.token_level
        rows = num_q_heads if self.qh else num_kv_heads
        # alpha-entmax instead of softmax over the selection (page level, per KV head)
        self.alpha = float(alpha)
        # Gaussian-aware adaptive selection per query head, attended with alpha-entmax
        self.gaussian = gaussian
        if gaussian and (page_size == 1 or self.alpha not in (1.5, 2.0) or per_query_head):
            raise ValueError("Gaussian-aware selection needs alpha 1.5 or 2 at the page level")
        self.entmax = self.alpha != 1.0 and not gaussian
        if self.entmax and (self.token_level or self.qh or not 1.0 < self.alpha <= 2.0):
            raise ValueError("entmax decoding needs 1 < alpha <= 2, page level, per-KV-head selection")
        if gaussian:
            topk = max(topk, 1)
        self.cache = PagedKVCache(num_blocks, num_kv_heads, page_size, head_dim, dtype, device,
                                  with_meta=not self.token_level, with_hh=self.token_level,
                                  with_std=gaussian)
        i32 = dict(dtype=torch.int32, device=device)
        self.block_table = torch.zeros((batch, bt_stride), **i32)
        self.seq_lens = torch.zeros((batch,), **i32)
        self.batch = make_batch(self.block_table, self.seq_lens)
        self.bt_stride = bt_stride
        self.max_pages = bt_stride
        if self.token_level:
            self.ret_cap = ret_cap
            self.ret_pos = torch.zeros((batch, num_kv_heads, ret_cap), **i32)
            self.ret_cnt = torch.zeros((batch, num_kv_heads), **i32)
            self.logits = torch.empty((batch, num_q_heads, ret_cap), dtype=torch.float32,
                                      device=device)
            self.evicted = torch.zeros((batch, num_kv_heads, ret_cap), **i32)
            self.evicted_cnt = torch.zeros((batch, num_kv_heads), **i32)
            self.sel_stride = ret_cap
        else:
            if topk <= 0:
                raise ValueError("page-level decoding needs topk >= 1")
            self.scores = torch.empty((batch, rows, bt_stride), dtype=torch.float32,
                                      device=device)
            self.sel_idx = torch.zeros((batch, rows, topk), **i32)
            self.sel_cnt = torch.zeros((batch, rows), **i32)
            self.sel_stride = topk
        self.out = torch.empty((batch, num_q_heads, head_dim), dtype=dtype, device=device)
        self.lse = torch.empty((batch, num_q_heads), dtype=torch.float32, device=device)
        self.workspace = alloc_decode_workspace(batch, rows if not self.token_level else num_kv_heads,
                                                num_q_heads, head_dim, page_size, self.sel_stride,
                                                device)
        if gaussian:
            # every page may qualify: selections as long as the table, one per query head
            self.sel_stride = bt_stride
            self.moments = torch.empty((batch, num_q_heads, bt_stride, 2), dtype=torch.float32,
                                       device=device)
            self.sel_idx = torch.zeros((batch, num_q_heads, bt_stride), **i32)
            self.sel_cnt = torch.zeros((batch, num_q_heads), **i32)
            self.tau_hat = torch.empty((batch, num_q_heads), dtype=torch.float32, device=device)
            self.tau = torch.empty((batch, num_q_heads), dtype=torch.float32, device=device)
            self.logits = torch.empty((batch, num_q_heads, bt_stride * page_size),
                                      dtype=torch.float32, device=device)
            self.ent_ws = alloc_entmax_workspace(batch, num_q_heads, num_q_heads, head_dim,
                                                 page_size, bt_stride, device)
        if self.entmax:
            self.ent_ws = alloc_entmax_workspace(batch, num_kv_heads, num_q_heads, head_dim,
                                                 page_size, self.sel_stride, device)
            self.tau = torch.empty((batch, num_q_heads), dtype=torch.float32, device=device)
            self.logits = torch.empty((batch, num_q_heads, self.sel_stride * page_size),
                                      dtype=torch.float32, device=device)
        self.dev_status = torch.zeros((1,), **i32)
        self.decode_cu = torch.arange(batch + 1, **i32)
        self.q_buf = torch.zeros((batch, num_q_heads, head_dim), dtype=dtype, device=device)
        self.k_buf = torch.zeros((batch, num_kv_heads, head_dim), dtype=dtype, device=device)
        self.v_buf = torch.zeros((batch, num_kv_heads, head_dim), dtype=dtype, device=device)
        self.graph = None

    # ------------------------------------------------------------------
    def set_block_table(self, bt: torch.Tensor):
        self.block_table.copy_(bt.to(device=self.device, dtype=torch.int32))

    def prefill(self, k: torch.Tensor, v: torch.Tensor, lens: Sequence[int]):
        """Append lens[b] tokens per request: k, v [sum(lens), H_kv, D] in request order.
        With proxy_prefill the retained lists take the tokens through the
        key-as-query absorb and eviction instead of all at once."""
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + int(n))
        new_cu = torch.tensor(cu, dtype=torch.int32, device=self.device)
        mx = max(int(n) for n in lens)
        if self.proxy_prefill:
            sa_append_kv(self.cache.struct, self.batch, k, v, new_cu, mx, hh=self.cache.hh,
                         dev_status=self.dev_status)
            sa_h2o_prefill(self.cache.struct, self.batch, new_cu, self.cache.hh,
                           self.cache.hh.shape[0], self.ret_pos, self.ret_cnt, self.ret_cap,
                           self.budget, self.n_sink, self.grace, self.decay, self.scale,
                           dev_status=self.dev_status)
        else:
            self._append(k, v, new_cu, mx)

    def _append(self, k, v, new_cu, max_new):
        if self.token_level:
            sa_append_kv(self.cache.struct, self.batch, k, v, new_cu, max_new, hh=self.cache.hh,
                         ret_pos=self.ret_pos, ret_cnt=self.ret_cnt, ret_cap=self.ret_cap,
                         dev_status=self.dev_status)
        else:
            sa_append_kv(self.cache.struct, self.batch, k, v, new_cu, max_new,
                         hh=self.cache.hh, dev_status=self.dev_status)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor):
        """One new token per request: k_new, v_new [B, H_kv, D]."""
        self._append(k_new, v_new, self.decode_cu, 1)

    def attend(self, q: torch.Tensor):
        """Attention of q [B, H_q, D] over the current cache (no append)."""
        if self.token_level:
            sa_sparse_decode(self.cache.struct, self.batch, q, self.H_q, self.ret_pos, self.ret_cnt,
                             self.ret_cap, self.scale, self.out, lse=self.lse, logits=self.logits,
                             logits_stride=self.ret_cap, workspace=self.workspace,
                             dev_status=self.dev_status)
            h2o = sa_h2o_update_window if self.window_softmax else sa_h2o_update
            h2o(self.batch, self.H_kv, self.H_q, self.logits, self.ret_cap, self.lse,
                          self.cache.hh, self.cache.hh.shape[0], self.ret_pos, self.ret_cnt,
                          self.ret_cap, self.budget, self.n_sink, self.grace, self.decay,
                          evicted=self.evicted, evicted_cnt=self.evicted_cnt,
                          dev_status=self.dev_status)
        elif self.gaussian:
            sa_gauss_select(self.cache.struct, self.batch, q, self.H_q, self.alpha, self.scale,
                            self.moments, self.max_pages, self.sel_idx, self.sel_cnt,
                            self.sel_stride, tau_hat=self.tau_hat, dev_status=self.dev_status)
            sa_sparse_decode_entmax_qh(self.cache.struct, self.batch, q, self.H_q, self.sel_idx,
                                       self.sel_cnt, self.sel_stride, self.alpha, self.scale,
                                       self.out, tau=self.tau, logits=self.logits,
                                       logits_stride=self.sel_stride * self.ps,
                                       workspace=self.ent_ws, dev_status=self.dev_status)
        elif self.qh:
            sa_score_pages_qh(self.cache.struct, self.batch, q, self.H_q, self.w_avg, self.w_peak,
                              self.scores, self.max_pages, dev_status=self.dev_status)
            sa_select_topk_reserved(self.scores, self.max_pages, self.batch, self.ps, self.H_q,
                                    self.topk, self.n_bos, self.n_eos, self.sel_idx, self.sel_cnt,
                                    dev_status=self.dev_status)
            sa_sparse_decode_qh(self.cache.struct, self.batch, q, self.H_q, self.sel_idx,
                                self.sel_cnt, self.topk, self.scale, self.out, lse=self.lse,
                                workspace=self.workspace, dev_status=self.dev_status)
        else:
            sa_score_pages(self.cache.struct, self.batch, q, self.H_q, self.w_avg, self.w_peak,
                           self.scores, self.max_pages, dev_status=self.dev_status)
            sa_select_topk_reserved(self.scores, self.max_pages, self.batch, self.ps, self.H_kv,
                                    self.topk, self.n_bos, self.n_eos, self.sel_idx, self.sel_cnt,
                                    dev_status=self.dev_status)
            if self.entmax:
                sa_sparse_decode_entmax(self.cache.struct, self.batch, q, self.H_q, self.sel_idx,
                                        self.sel_cnt, self.topk, self.alpha, self.scale, self.out,
                                        tau=self.tau, logits=self.logits,
                                        logits_stride=self.topk * self.ps, workspace=self.ent_ws,
                                        dev_status=self.dev_status)
                return self.out
            sa_sparse_decode(self.cache.struct, self.batch, q, self.H_q, self.sel_idx,
                             self.sel_cnt, self.topk, self.scale, self.out, lse=self.lse,
                             workspace=self.workspace, dev_status=self.dev_status)
        return self.out

    def step(self, q: torch.Tensor, k_new: Optional[torch.Tensor] = None,
             v_new: Optional[torch.Tensor] = None):
        if self.token_level or self.qh or self.entmax or self.gaussian:
            if k_new is not None:
                self.append(k_new, v_new)
            return self.attend(q)
        sa_decode_step(self.cache.struct, self.batch, k_new, v_new,
                       self.decode_cu if k_new is not None else None,
                       1 if k_new is not None else 0, q, self.H_q, self.w_avg, self.w_peak,
                       self.scores, self.max_pages, self.topk, self.sel_idx, self.sel_cnt,
                       self.scale, self.out, lse=self.lse, workspace=self.workspace,
                       dev_status=self.dev_status, n_bos=self.n_bos, n_eos=self.n_eos)
        return self.out

    # ------------------------------------------------------------------
    def capture(self, append: bool = True):
        """Record one step (reading q_buf / k_buf / v_buf) into a CUDA graph."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.step(self.q_buf, self.k_buf if append else None, self.v_buf if append else None)
        torch.cuda.current_stream(self.device).wait_stream(s)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()
        return self.out
