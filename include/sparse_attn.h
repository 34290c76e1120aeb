/*
 * sparse_attn.h -- C ABI of the GB300 (sm_103a) page-selected sparse decode
 * library (libsparse_attn / _sparse_attn.so).
 *
 * One decode step of page-selected sparse attention over a paged KV cache:
 *   sa_append_kv      write new keys/values, refresh the written pages'
 *                     element-wise key statistics, zero their H2O slots
 *   sa_score_pages    score every page per KV head from the statistics
 *   sa_select_topk    top-k pages per KV head, the tail page always kept
 *   sa_sparse_decode  exact softmax attention over the selected pages only,
 *                     split across pages, partials merged by log-sum-exp
 *   sa_h2o_update     token-level (page_size 1) decayed heavy-hitter fold and
 *                     sink/grace-protected eviction
 *   sa_decode_step    the page-level chain (append, score, select, decode) in
 *                     one call, kernels overlapped by programmatic launch
 *   sa_select_topk_reserved, sa_h2o_update_window
 *                     the selection and the H2O fold with reserved leading and
 *                     trailing pages / tokens
 *   sa_score_pages_qh, sa_sparse_decode_qh
 *                     scores, selection and attention per query head
 *   sa_h2o_prefill    H2O absorb / eviction of appended tokens with the new key
 *                     as the query (prefill side)
 *   sa_sparse_decode_entmax, sa_sparse_decode_entmax_qh, sa_entmax_workspace_size
 *                     attention over the selection with alpha-entmax
 *   sa_gauss_select   Gaussian-aware adaptive page selection per query head
 *   sa_shard_lengths, sa_shard_selection, sa_merge_states
 *                     sequence sharding: page ranges per shard, merged states
 *
 * Sources (cited by page title and section):
 *   [vortex]  "flow: add H2O sparse attention (page-level and token-level,
 *             MHA + GQA)", vortex_torch pull request 6.
 *   [velox]   "H2O -- Cumulative Attention-Mass Heavy-Hitter Oracle
 *             Eviction", VeloxQuant-MLX docs.
 *   [vllmcpp] "test_ops_mla_chunked_context.cpp", vllm.cpp tests.
 *   [entmax]  "EntmaxKV" README.
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership: the caller owns every buffer. All array pointers are DEVICE
 *   pointers (CUDA global memory of the current device) unless marked "host".
 *   Struct arguments themselves are read on the host during the call and may
 *   be freed when it returns. The library never allocates device memory;
 *   scratch comes from a caller-provided workspace.
 * Asynchrony: every call only enqueues work on `stream` (a cudaStream_t
 *   passed as void*; NULL = the legacy default stream) and returns; nothing
 *   synchronises. Results are visible in stream order.
 * Host errors: arguments are validated before anything is launched; a
 *   violation returns SA_ERR_INVALID_ARG / SA_ERR_UNSUPPORTED /
 *   SA_ERR_WORKSPACE and launches nothing. A failed launch returns
 *   SA_ERR_CUDA.
 * Data errors: faults that only the data reveals (a block-table entry outside
 *   [0, num_blocks), a page index outside the request, a full retained list)
 *   never trap. The kernel sets sticky bits in the caller's int32 status word
 *   `dev_status` (nullable: then not recorded), skips the bad unit's memory
 *   access, and finishes; the caller reads the word when convenient.
 * Alignment: the pools (k, v, meta, kstd) and q start on 16-byte boundaries
 *   (the kernels read them in 16-byte units); a misaligned one is rejected
 *   with SA_ERR_INVALID_ARG.
 * Layout: pools are [num_blocks, num_kv_heads, page_size, head_dim] (one
 *   contiguous (block, head) tile), row-major; this differs from vLLM's
 *   [2, num_blocks, page_size, H_kv, D] (cited by [entmax] "How it works")
 *   only in the order of the middle axes. Logical page p of request b lives in
 *   block block_table[b * bt_stride + p]; position j is page j / page_size,
 *   slot j % page_size. Query head g' belongs to KV head g' / G with
 *   G = num_q_heads / num_kv_heads.
 * Supported: dtype bf16 or fp16; head_dim 64 or 128; page_size a power of two
 *   in [1, 128]; G in [1, 16].
 */
#ifndef SPARSE_ATTN_H_
#define SPARSE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sa_status {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1,   /* a null required pointer, a bad size or a broken constraint */
  SA_ERR_UNSUPPORTED = 2,   /* a valid configuration the library does not implement */
  SA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than sa_decode_workspace_size() */
  SA_ERR_CUDA = 4           /* a CUDA launch or runtime call failed */
} sa_status;

typedef enum sa_dtype { SA_BF16 = 0, SA_FP16 = 1 } sa_dtype;

/* Sticky bits of the device status word. */
#define SA_DEV_BAD_BLOCK 1  /* block-table entry outside [0, num_blocks), or page index out of range */
#define SA_DEV_OVERFLOW 2   /* table or retained-list capacity exceeded; the excess was dropped */
#define SA_DEV_BAD_COUNT 4  /* a selection / retained count outside [0, stride] (clamped) */
#define SA_DEV_TIMEOUT 8    /* a bounded wait inside a kernel gave up (the kernel stopped early) */

/* The paged cache: pools plus per-page statistics. */
typedef struct sa_cache {
  void* k;              /* [num_blocks, num_kv_heads, page_size, head_dim], dtype */
  void* v;              /* same layout as k */
  void* meta;           /* [num_blocks, num_kv_heads, 3, head_dim], dtype: rows (k_min, k_max,
                           k_mean) of the page's valid tokens; may be NULL where no call needs it */
  int32_t dtype;        /* sa_dtype */
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t page_size;
  int32_t head_dim;
  void* kstd;           /* nullable [num_blocks, num_kv_heads, head_dim], dtype: k_std, the
                           population standard deviation of each dimension over the page's
                           valid tokens (for sa_gauss_select); refreshed by sa_append_kv when
                           present */
} sa_cache;

/* The batch: block table and lengths. */
typedef struct sa_batch {
  const int32_t* block_table;  /* [batch, bt_stride]: logical page -> physical block */
  int32_t* seq_lens;           /* [batch]: cached tokens per request; advanced only by sa_append_kv */
  int32_t batch;
  int32_t bt_stride;           /* table row length = page capacity per request */
} sa_batch;

/*
 * sa_append_kv -- append new tokens and refresh the statistics of every page
 * they touch.
 *
 * [vortex] "Page-level variants" and "Token-level variants" point 2:
 * k_min / k_max / k_mean are overwriting reductions recomputed over a written
 * page, and hh_score of the written pages is reset to zero because a recycled
 * pool page keeps stale contents. [entmax] "How it works" / "Quick start":
 * the decode call appends k_new / v_new and refreshes per-page key statistics.
 *
 * Request b's new tokens are rows new_cu[b] .. new_cu[b+1]-1 of k_new / v_new
 * ([T_total, num_kv_heads, head_dim], dtype) and go to positions
 * seq_lens[b] .. seq_lens[b] + n_b - 1. For every page touched, each KV head's
 * statistics are recomputed over the page's valid tokens only (old tokens read
 * from the pool, stale slots past the new length never read): k_min and k_max
 * exactly, k_mean as the float64 mean rounded once (to nearest even) to dtype.
 * Written if cache->meta != NULL.
 *   new_cu            [batch + 1] int32, device, non-decreasing, new_cu[0] = 0
 *   max_new_per_req   host: an upper bound on any n_b (sizes the grid); n_b above
 *                     it sets SA_DEV_OVERFLOW and the excess is dropped
 *   hh                nullable bf16 [num_blocks * page_size, num_kv_heads]: the
 *                     H2O score of token slot (block * page_size + slot); the
 *                     slots written here are set to 0
 *   ret_pos, ret_cnt  nullable (both or neither): token-level retained lists
 *                     [batch, num_kv_heads, ret_cap] int32 positions, ascending,
 *                     and their counts [batch, num_kv_heads]; the new positions
 *                     are appended to every KV head's list
 * Finally seq_lens[b] += n_b (and ret_cnt += n_b), after all reads of the old
 * values. A position beyond bt_stride * page_size, or a list beyond ret_cap,
 * sets SA_DEV_OVERFLOW and is dropped.
 */
sa_status sa_append_kv(const sa_cache* cache, const sa_batch* batch, const void* k_new,
                       const void* v_new, const int32_t* new_cu, int32_t max_new_per_req,
                       void* hh, int32_t* ret_pos, int32_t* ret_cnt, int32_t ret_cap,
                       int32_t* dev_status, void* stream);

/*
 * sa_score_pages -- score every cached page of every (request, KV head).
 *
 * [vortex] "Page-level variants": average relevance q . mean(k) and the peak
 * relevance envelope bound sum_d max(q_d * max_d, q_d * min_d) >= max_k q . k
 * (both envelopes, since q is signed), combined as w_avg * avg + w_peak * peak
 * (the Add(alpha = w_avg, beta = w_peak) of the page); [entmax] "How it works"
 * (scored from page statistics without touching the cached tokens). The G
 * query heads of a KV head are reduced to one ranking by the mean of their
 * scores; no softmax scale is applied.
 *   q        [batch, num_q_heads, head_dim], dtype
 *   scores   [batch, num_kv_heads, max_pages] float32; entry (b, h, p) is
 *            written for p < ceil(seq_lens[b] / page_size), others untouched
 *   max_pages  host: row length of scores, >= every request's page count
 *            (else SA_DEV_OVERFLOW for that request)
 * A page whose block id is out of range scores NaN and sets SA_DEV_BAD_BLOCK.
 * Needs cache->meta. Limits: batch <= 1024 (else SA_ERR_UNSUPPORTED). Arithmetic: float32, using the exact identity
 * max(q*M, q*m) = max(q,0)*M + min(q,0)*m (M >= m) so the cost per page does
 * not grow with G.
 */
sa_status sa_score_pages(const sa_cache* cache, const sa_batch* batch, const void* q,
                         int32_t num_q_heads, float w_avg, float w_peak, float* scores,
                         int32_t max_pages, int32_t* dev_status, void* stream);

/*
 * sa_score_pages_qh -- sa_score_pages with one score row per query head.
 *
 * [entmax] "How it works", "Top-k": pages are ranked for each query head and
 * the top pages are kept per query head. Each query head g of KV head h = g / G
 * scores the pages of h from their statistics alone (no reduction over the
 * group): S_g(p) = sum_d [w_avg q_gd mean_pd + w_peak max(q_gd max_pd, q_gd min_pd)].
 *   scores   [batch, num_q_heads, max_pages] float32 (entries past a
 *            request's page count untouched)
 * Everything else as sa_score_pages. The rows select with sa_select_topk /
 * sa_select_topk_reserved called with num_kv_heads = num_q_heads, and
 * sa_sparse_decode_qh attends them.
 */
sa_status sa_score_pages_qh(const sa_cache* cache, const sa_batch* batch, const void* q,
                            int32_t num_q_heads, float w_avg, float w_peak, float* scores,
                            int32_t max_pages, int32_t* dev_status, void* stream);

/*
 * sa_select_topk -- top-k pages per (request, KV head), tail page forced.
 *
 * [entmax] "How it works", "Top-k": keep topk pages, the budget counting the
 * always-attended tail page. With n = ceil(seq_lens[b] / page_size): if
 * n <= topk every page is selected; otherwise page n-1 plus the topk-1 best of
 * pages 0..n-2 by (score descending, page index ascending), -0 equal to +0,
 * NaN after every number. Output indices ascending.
 *   scores   [batch, num_kv_heads, max_pages] float32 (from sa_score_pages)
 *   sel_idx  [batch, num_kv_heads, topk] int32; entries past sel_cnt untouched
 *   sel_cnt  [batch, num_kv_heads] int32 = min(topk, n)
 * Limits: max_pages <= 45056 (the candidate keys of one (request, KV head)
 * are held in shared memory), else SA_ERR_UNSUPPORTED.
 */
sa_status sa_select_topk(const float* scores, int32_t max_pages, const sa_batch* batch,
                         int32_t page_size, int32_t num_kv_heads, int32_t topk,
                         int32_t* sel_idx, int32_t* sel_cnt, int32_t* dev_status,
                         void* stream);

/*
 * sa_select_topk_reserved -- sa_select_topk with reserved leading and
 * trailing pages.
 *
 * [vortex] follow-up comment ("Two things I had to fix"): the first
 * page_reserved_bos and the last page_reserved_eos pages are kept
 * unconditionally and top-k ranks only the window between them. The reserved
 * pages count against the budget (as [entmax] "Top-k" counts the tail page):
 * with n = ceil(seq_lens[b] / page_size), n <= topk selects every page;
 * otherwise pages 0 .. n_bos-1, pages n-n_eos .. n-1 and the
 * topk - n_bos - n_eos best of pages n_bos .. n-n_eos-1 by (score descending,
 * page index ascending), -0 equal to +0, NaN after every number; indices
 * ascending, sel_cnt = min(topk, n). n_bos = 0, n_eos = 1 is sa_select_topk.
 * Constraints: n_bos >= 0, n_eos >= 1 (the tail page, which the attention
 * needs), n_bos + n_eos <= topk (else SA_ERR_INVALID_ARG).
 */
sa_status sa_select_topk_reserved(const float* scores, int32_t max_pages, const sa_batch* batch,
                                  int32_t page_size, int32_t num_kv_heads, int32_t topk,
                                  int32_t n_bos, int32_t n_eos, int32_t* sel_idx, int32_t* sel_cnt,
                                  int32_t* dev_status, void* stream);

/*
 * sa_decode_workspace_size -- bytes of workspace sa_sparse_decode needs for
 * these sizes (host function, no GPU access). The workspace holds the split
 * partial states and one ticket counter per (request, KV head); it must be
 * zero-filled once before its first use (sa_decode_workspace_init does this)
 * and every call leaves the counters at zero again. Calls that share a
 * workspace must be ordered on one stream.
 */
size_t sa_decode_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t num_q_heads,
                                int32_t head_dim, int32_t page_size, int32_t sel_stride);

/* Zero-fill a decode workspace on `stream` (cudaMemsetAsync; allocates nothing). */
sa_status sa_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * sa_sparse_decode -- exact softmax attention of each query head over the
 * valid tokens of its KV head's selected pages.
 *
 * [entmax] "How it works": only the selected pages are attended and the
 * attention is exact over that selection. [vortex] "Token-level variants"
 * point 1: the softmax scale defaults to head_dim ** -0.5. [vllmcpp] the
 * chunked loop must equal single-shot attention: the selected tokens are split
 * across CTAs, each emits a partial (o_s, lse_s) (lse_s = -inf when empty),
 * and the partials are merged exactly: lse = log sum_s exp(lse_s),
 * o = sum_s exp(lse_s - lse) o_s; no tokens at all gives o = 0, lse = -inf.
 *   q          [batch, num_q_heads, head_dim], dtype
 *   sel_idx    [batch, num_kv_heads, sel_stride] int32 logical page indices
 *              (for page_size 1: token positions), sel_cnt [batch, num_kv_heads];
 *              the selection may be in any order; entries are visited in order
 *   scale      softmax scale; <= 0 selects head_dim ** -0.5
 *   out        [batch, num_q_heads, head_dim], dtype
 *   lse        nullable float32 [batch, num_q_heads], natural log
 *   logits     nullable float32 [batch, num_q_heads, logits_stride]: the scaled
 *              logit scale * q . k of selection token i = e * page_size + slot
 *              (entry e, slot within the page); -inf for slots past the page's
 *              fill and for entries skipped as invalid; logits_stride >=
 *              sel_stride * page_size
 *   workspace  see sa_decode_workspace_size
 * Only the valid tokens of each selected page are read (the tail page's stale
 * slots are zero-filled in shared memory, never loaded). Tensor cores
 * (mma.sync bf16/fp16, float32 accumulate) compute q.K and P.V; softmax in
 * float32. Selected pages whose block id is out of range are skipped with
 * SA_DEV_BAD_BLOCK.
 */
sa_status sa_sparse_decode(const sa_cache* cache, const sa_batch* batch, const void* q,
                           int32_t num_q_heads, const int32_t* sel_idx, const int32_t* sel_cnt,
                           int32_t sel_stride, float scale, void* out, float* lse,
                           float* logits, int32_t logits_stride, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * sa_sparse_decode_qh -- sa_sparse_decode with a selection per query head.
 *
 * [entmax] "Top-k" (pages kept per query head) and "How it works" (exact
 * attention over the selection): query head g attends exactly the pages its
 * own row lists, of its KV head g / G.
 *   sel_idx  [batch, num_q_heads, sel_stride] int32, sel_cnt [batch, num_q_heads]
 *   workspace  sa_decode_workspace_size(batch, num_q_heads, num_q_heads,
 *            head_dim, page_size, sel_stride) bytes (each query head a unit
 *            of one head)
 * q, out, lse, scale and the error behaviour as sa_sparse_decode; no logits.
 */
sa_status sa_sparse_decode_qh(const sa_cache* cache, const sa_batch* batch, const void* q,
                              int32_t num_q_heads, const int32_t* sel_idx, const int32_t* sel_cnt,
                              int32_t sel_stride, float scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream);

/*
 * sa_entmax_workspace_size -- bytes of workspace sa_sparse_decode_entmax
 * needs for these sizes (host function; reads the device's SM count). The
 * workspace holds the logits (when the caller passes none), the per-split
 * partial sums and one counter per (request, KV head); it must be zero-filled
 * once before its first use (sa_decode_workspace_init does this) and every
 * call leaves the counters at zero again. Calls that share a workspace must be
 * ordered on one stream.
 */
size_t sa_entmax_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t num_q_heads,
                                int32_t head_dim, int32_t page_size, int32_t sel_stride);

/*
 * sa_sparse_decode_entmax -- attention over the selected pages with
 * alpha-entmax in place of the softmax.
 *
 * [entmax] "How it works" and "Quick start": the selection of sa_select_topk
 * is attended exactly, normalised by alpha-entmax (the pages' default
 * alpha = 1.5; alpha = 2 is sparsemax). With z_j = scale * q . k_j over the
 * valid tokens of the selection and a_j = (alpha - 1) z_j,
 *   p_j = max(a_j - tau, 0) ^ (1 / (alpha - 1)),  sum_j p_j = 1,
 *   o   = sum_j p_j v_j.
 * tau is computed in float32: for alpha = 1.5 and 2 as the closed form on the
 * support (the largest set whose threshold stays below its smallest member,
 * found by Newton's method from max_j a_j - 1), otherwise by Newton's method
 * until its step falls below float32 resolution.
 *   q, sel_idx, sel_cnt, sel_stride, scale, out   as sa_sparse_decode
 *   alpha      1 < alpha <= 2, else SA_ERR_INVALID_ARG
 *   tau        nullable float32 [batch, num_q_heads]: the threshold in units
 *              of a; NaN for a head with no valid token (its output is 0)
 *   logits     nullable float32 [batch, num_q_heads, logits_stride], as
 *              sa_sparse_decode's (logits_stride >= sel_stride * page_size)
 *   workspace  sa_entmax_workspace_size(...) bytes, else SA_ERR_WORKSPACE
 * The output is divided by the float32 sum of the p_j it used (1 up to the
 * rounding of tau). K of every selected token is read once; V only for the
 * tokens some query head of the group keeps. Limits: num_q_heads / num_kv_heads
 * <= 16, and the selection entries one CTA resolves must fit its shared
 * memory (a few thousand entries), else SA_ERR_UNSUPPORTED before anything is
 * launched. Data errors as sa_sparse_decode.
 */
sa_status sa_sparse_decode_entmax(const sa_cache* cache, const sa_batch* batch, const void* q,
                                  int32_t num_q_heads, const int32_t* sel_idx,
                                  const int32_t* sel_cnt, int32_t sel_stride, float alpha,
                                  float scale, void* out, float* tau, float* logits,
                                  int32_t logits_stride, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream);

/*
 * sa_sparse_decode_noalloc -- sa_sparse_decode without a caller workspace.
 *
 * No counterpart on the pages: this is an integration convenience. Some
 * callers cannot allocate device memory where they call the decode -- a plugin
 * handed fixed buffers by a host engine, a runtime whose memory plan is frozen
 * after start-up, a real-time loop that must never enter the allocator. This
 * entry point allocates nothing: the split partials and tickets live in one
 * fixed device array inside the library, of sa_sparse_decode_noalloc_capacity()
 * bytes (4 MiB), which every GPU that loads the library keeps until the
 * process exits. Arguments, layouts and results are those of
 * sa_sparse_decode; the caller still passes every input and output.
 *   - A call whose sizes need more scratch than the capacity (see
 *     sa_decode_workspace_size) returns SA_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call resets the tickets it uses with cudaMemsetAsync on `stream`.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and corrupt each other's results; order
 *     them on one stream.
 */
sa_status sa_sparse_decode_noalloc(const sa_cache* cache, const sa_batch* batch, const void* q,
                                   int32_t num_q_heads, const int32_t* sel_idx,
                                   const int32_t* sel_cnt, int32_t sel_stride, float scale,
                                   void* out, float* lse, float* logits, int32_t logits_stride,
                                   int32_t* dev_status, void* stream);

/* Bytes of the fixed scratch array sa_sparse_decode_noalloc uses (host function). */
size_t sa_sparse_decode_noalloc_capacity(void);

/*
 * sa_h2o_update -- token-level H2O: fold this step's attention probabilities
 * into the bf16 heavy-hitter scores and evict above budget (page_size 1).
 *
 * [vortex] "Token-level variants" points 1 and 3: the accumulated quantity is
 * the softmax probability (not the logit), hh_score is bf16 and decays,
 * out = 1 * attn + decay * old. [velox] "Parameters" and "How it works": the
 * first n_sink retained tokens and the newest `grace` are never evicted;
 * while more than `budget` tokens remain the lowest-scoring eligible one is
 * removed (ties to the lowest position); afterwards at most `budget` remain.
 * For every retained entry j of (b, h) (position ret_pos[b, h, j]):
 *   p_bar_j = (1/G) sum_g exp(logits[b, h*G+g, j] - lse[b, h*G+g])   (float32)
 *   hh[slot_j, h] = bf16(decay * hh[slot_j, h] + p_bar_j)   (float64 fma, one rounding)
 * with slot_j = block_table[b, pos_j] (page_size 1); then the eviction, which
 * compacts ret_pos in place (order kept) and sets ret_cnt.
 *   logits, lse  from sa_sparse_decode over sel_idx = ret_pos, sel_cnt = ret_cnt
 *   hh           bf16 [num_slots, num_kv_heads], num_slots = blocks of the pool
 *   evicted      nullable int32 [batch, num_kv_heads, ret_cap]: evicted positions,
 *                ascending; evicted_cnt nullable int32 [batch, num_kv_heads]
 * Constraints: budget > n_sink + grace (as [velox] requires), 0 < decay <= 1,
 * ret_cap <= 32768.
 */
sa_status sa_h2o_update(const sa_batch* batch, int32_t num_kv_heads, int32_t num_q_heads,
                        const float* logits, int32_t logits_stride, const float* lse, void* hh,
                        int32_t num_slots, int32_t* ret_pos, int32_t* ret_cnt, int32_t ret_cap,
                        int32_t budget, int32_t n_sink, int32_t grace, float decay,
                        int32_t* evicted, int32_t* evicted_cnt, int32_t* dev_status,
                        void* stream);

/*
 * sa_decode_step -- one whole page-level decode step in one call:
 * sa_append_kv, sa_score_pages, sa_select_topk, sa_sparse_decode.
 *
 * [vortex] "Page-level variants" and [entmax] "How it works": the new token's
 * key refreshes its page's statistics, every page is scored from the
 * statistics, the top-k pages (tail forced) are chosen and attention runs
 * exactly over them. Arguments mean what they mean in the four calls (the
 * selection row length is topk; no H2O slots, no retained lists, no logits);
 * the selection is sa_select_topk_reserved's with n_bos, n_eos (0, 1 gives
 * sa_select_topk's).
 *   k_new      nullable: NULL (or max_new_per_req 0) skips the append, and
 *              v_new / new_cu are then ignored
 *   workspace  at least sa_decode_workspace_size(batch, num_kv_heads,
 *              num_q_heads, head_dim, page_size, topk) bytes, zero-filled once
 *              (else SA_ERR_WORKSPACE)
 * Needs cache->meta. Limits: those of the four calls.
 * The kernels are chained by programmatic dependent launch on `stream`: each
 * one starts its prologue (reading q, setting up barriers) while its
 * predecessor finishes and waits on the device for the data it consumes.
 * With max_new_per_req == 1 the append runs beside the scorer, which then
 * scores the lengths from before the append: every page the append leaves
 * untouched gets its exact score, while the score entry of the page the new
 * token went to (the tail, always selected) is unspecified. With
 * max_new_per_req > 1 the append runs first and every score is exact.
 * Selection, output and lse are those of the four calls in order.
 */
sa_status sa_decode_step(const sa_cache* cache, const sa_batch* batch, const void* k_new,
                         const void* v_new, const int32_t* new_cu, int32_t max_new_per_req,
                         const void* q, int32_t num_q_heads, float w_avg, float w_peak,
                         float* scores, int32_t max_pages, int32_t topk, int32_t n_bos,
                         int32_t n_eos, int32_t* sel_idx, int32_t* sel_cnt, float scale,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         int32_t* dev_status, void* stream);

/*
 * sa_h2o_update_window -- sa_h2o_update with the reserved windows of [vortex]
 * (follow-up comment, "Two things I had to fix"): hh_score stays zero on the
 * reserved tokens and the softmax is normalised over the window between them.
 * Here the reserved entries are the protected ones, the first n_sink and the
 * last grace entries of the retained list: they receive p_bar = 0, and for the
 * entries j in between
 *   p_bar_j = (1/G) sum_g exp(logits[g, j] - lse'_g),
 *   lse'_g  = log sum over those entries of exp(logits[g, .])   (float32);
 * lse is not read. Eviction and every other argument as sa_h2o_update;
 * G <= 16.
 */
sa_status sa_h2o_update_window(const sa_batch* batch, int32_t num_kv_heads, int32_t num_q_heads,
                               const float* logits, int32_t logits_stride, const float* lse,
                               void* hh, int32_t num_slots, int32_t* ret_pos, int32_t* ret_cnt,
                               int32_t ret_cap, int32_t budget, int32_t n_sink, int32_t grace,
                               float decay, int32_t* evicted, int32_t* evicted_cnt,
                               int32_t* dev_status, void* stream);

/*
 * sa_h2o_prefill -- H2O absorb and eviction for newly appended tokens, each
 * token's own key standing in for its query (page_size 1, bf16 pool).
 *
 * [velox] "How it works": for every incoming token, per head, the new key k
 * attends to every stored key, attn = softmax(K k * scale); stored scores
 * become scores * decay + attn; the new token starts at 0; while more than
 * budget entries remain, the lowest (score, position) entry outside the first
 * n_sink and the newest grace list entries is removed. The batched absorb of
 * velox's changelog is the same arithmetic as this token-by-token loop.
 * Request b's new tokens are positions seq_lens[b] - n_b .. seq_lens[b] - 1
 * with n_b = new_cu[b+1] - new_cu[b] (already written by sa_append_kv, without
 * retained lists); they are processed in order against the retained list
 * (ret_pos / ret_cnt, at most budget entries, every position below them).
 * Scores: bf16 in hh [num_slots, num_kv_heads] (slot = block of the position),
 * each fold decay * hh + attn one float64 fma rounded once; attn in float32.
 *   scale      <= 0 selects head_dim ** -0.5
 *   evicted    nullable int32 [batch, num_kv_heads, evicted_cap]: positions
 *              evicted, in eviction order; evicted_cnt [batch, num_kv_heads]
 * Limits: budget + 1 <= 1024 and the retained keys of a (request, KV head)
 * fit in shared memory (budget <= 700 at head_dim 128), else
 * SA_ERR_UNSUPPORTED. One CTA per (request, KV head) holds its keys on chip
 * for the whole call.
 */
sa_status sa_h2o_prefill(const sa_cache* cache, const sa_batch* batch, const int32_t* new_cu,
                         void* hh, int32_t num_slots, int32_t* ret_pos, int32_t* ret_cnt,
                         int32_t ret_cap, int32_t budget, int32_t n_sink, int32_t grace,
                         float decay, float scale, int32_t* evicted, int32_t* evicted_cnt,
                         int32_t evicted_cap, int32_t* dev_status, void* stream);

/*
 * sa_sparse_decode_entmax_qh -- sa_sparse_decode_entmax with a selection per
 * query head.
 *
 * [entmax] "How it works" (pages kept per query head; the selected pages
 * attended exactly with alpha-entmax): query head g attends the pages of its
 * own row, of its KV head g / G.
 *   sel_idx  [batch, num_q_heads, sel_stride] int32, sel_cnt [batch, num_q_heads]
 *   workspace  sa_entmax_workspace_size(batch, num_q_heads, num_q_heads,
 *            head_dim, page_size, sel_stride) bytes (each query head a unit of
 *            one head), zero-filled once
 * Everything else as sa_sparse_decode_entmax.
 */
sa_status sa_sparse_decode_entmax_qh(const sa_cache* cache, const sa_batch* batch, const void* q,
                                     int32_t num_q_heads, const int32_t* sel_idx,
                                     const int32_t* sel_cnt, int32_t sel_stride, float alpha,
                                     float scale, void* out, float* tau, float* logits,
                                     int32_t logits_stride, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * sa_gauss_select -- Gaussian-aware page selection, one selection per query
 * head.
 *
 * [entmax] "How it works" (Gaussian-aware strategy): each page's scores are
 * modelled as a Gaussian from the per-page k_mean and k_std (without touching
 * the cached tokens), the distributional entmax constraint is solved for the
 * threshold tau_hat (one Gaussian for the whole context: heads without ALiBi),
 * and every page whose estimated maximum can cross tau_hat is selected; the
 * count adapts to the score distribution. With z = scale * q . k, f_p the
 * page's valid tokens and the page's dimensions taken as independent:
 *   m_p = scale sum_d q_d mean_pd,  v_p = scale^2 sum_d q_d^2 std_pd^2
 *   N = sum f_p, M = sum f m / N, V = sum f (v + m^2) / N - M^2
 *   tau_hat: N E[((alpha - 1) Z - tau_hat)_+ ^ (1 / (alpha - 1))] = 1, Z ~ N(M, V)
 *   keep p  iff (alpha - 1)(m_p + sqrt(2 ln f_p) sqrt(v_p)) > tau_hat, or p is
 *           the tail page (sqrt(2 ln f) bounds the expected maximum of f
 *           Gaussian scores)
 *   q        [batch, num_q_heads, head_dim], dtype
 *   alpha    1.5 or 2 (the closed forms of the truncated moments), else
 *            SA_ERR_UNSUPPORTED
 *   scale    <= 0 selects head_dim ** -0.5
 *   moments  float32 scratch [batch, num_q_heads, max_pages, 2] (m_p, v_p)
 *   max_pages >= batch->bt_stride; sel_stride >= max_pages
 *   sel_idx  [batch, num_q_heads, sel_stride] int32, ascending; sel_cnt
 *            [batch, num_q_heads] (0 for an empty request)
 *   tau_hat  nullable float32 [batch, num_q_heads] (in units of (alpha - 1) z)
 * Needs cache->meta (k_mean) and cache->kstd, both refreshed by sa_append_kv.
 * Pages whose block id is out of range are never kept (except the tail, left
 * to the decode's own check) and set SA_DEV_BAD_BLOCK; a request with more
 * pages than bt_stride sets SA_DEV_OVERFLOW and is read up to its row's end.
 * bf16 caches run m_p and v_p on the tensor cores (the squares split exactly
 * into two bf16 terms, every product exact, float32 sums); fp16 caches in
 * float32 FMAs. The selection feeds
 * sa_sparse_decode_entmax_qh, whose tau is exact over the selected tokens.
 */
sa_status sa_gauss_select(const sa_cache* cache, const sa_batch* batch, const void* q,
                          int32_t num_q_heads, float alpha, float scale, float* moments,
                          int32_t max_pages, int32_t* sel_idx, int32_t* sel_cnt,
                          int32_t sel_stride, float* tau_hat, int32_t* dev_status, void* stream);

/*
 * Sequence sharding -- the pages of every request split into contiguous
 * ranges [page_lo, page_hi) held by different shards (devices).
 *
 * [vllmcpp] MergeAttnStates: attention over a split of the keys is exact once
 * the partial states are merged by log-sum-exp. [entmax] "Top-k": the
 * selection is over the whole request, tail forced. A sharded step: each
 * shard computes the lengths of its range (sa_shard_lengths), scores its
 * pages with sa_score_pages on a batch view (block_table + page_lo, the same
 * bt_stride, its lengths), the score slices are gathered into one row per
 * (request, KV head) (the exchange), one sa_select_topk runs over the whole
 * rows, each shard takes its part of the selection (sa_shard_selection) and
 * attends it with sa_sparse_decode (o and lse), and the parts are merged by
 * sa_merge_states. Appends are not sharded here.
 *
 * sa_shard_lengths: shard_lens[b] = clamp(seq_lens[b] - page_lo * page_size,
 *   0, (page_hi - page_lo) * page_size); device arrays [batch] int32.
 * sa_shard_selection: for each of num_units rows of sel_idx [num_units,
 *   sel_stride] (counts sel_cnt), the entries with page_lo <= p < page_hi as
 *   p - page_lo, in order, into shard_idx [num_units, shard_stride] and
 *   shard_cnt; entries beyond shard_stride set SA_DEV_OVERFLOW.
 * sa_merge_states: o_parts [num_shards, rows, head_dim] (dtype), lse_parts
 *   [num_shards, rows] float32 (natural log; -inf for an empty part) ->
 *   out [rows, head_dim] (dtype) and lse (nullable) [rows]; +inf and NaN
 *   count as empty parts. A row whose parts are all empty would be 0/0:
 *   as in the MergeAttnStates test's reference, it takes the prefix (part
 *   0) output and lse = -inf (a sa_sparse_decode part with no keys holds
 *   o = 0, so an empty request still merges to 0).
 */
sa_status sa_shard_lengths(const int32_t* seq_lens, int32_t batch, int32_t page_size, int32_t page_lo,
                           int32_t page_hi, int32_t* shard_lens, void* stream);
sa_status sa_shard_selection(const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_stride,
                             int32_t num_units, int32_t page_lo, int32_t page_hi, int32_t* shard_idx,
                             int32_t* shard_cnt, int32_t shard_stride, int32_t* dev_status,
                             void* stream);
sa_status sa_merge_states(const void* o_parts, const float* lse_parts, int32_t num_shards, int32_t rows,
                          int32_t head_dim, int32_t dtype, void* out, float* lse, void* stream);

/*
 * Self-test of the bounded in-kernel wait (no counterpart on the pages: it
 * checks this library's "Bad data" contract -- every wait inside a kernel
 * gives up after a time limit, sets SA_DEV_TIMEOUT in the caller's status
 * word and lets the kernel return, so the context stays usable).
 *
 * One warp waits, through the wait the library's kernels use, on an mbarrier
 * that expects two arrivals and receives `arrivals` (0, 1 or 2) of them,
 * giving up after limit_ns (0 < limit_ns <= 100 ms) instead of the default
 * ~1 s. arrivals = 2: the wait completes, *result = 1, dev_status unchanged.
 * arrivals < 2: the wait runs out, *result = 0 and SA_DEV_TIMEOUT is set.
 * dev_status, result: device int32 (caller-owned). Asynchronous on `stream`;
 * SA_ERR_INVALID_ARG for other arguments, nothing launched.
 */
sa_status sa_wait_selftest(int32_t arrivals, int64_t limit_ns, int32_t* dev_status, int32_t* result,
                           void* stream);

/* Human-readable name of a status code (static string). */
const char* sa_status_string(sa_status status);

/* Library version, e.g. "0.1.0" (static string). */
const char* sa_version(void);

/* sizeof(sa_cache) (which = 0) or sizeof(sa_batch) (which = 1) as built, so a
 * binding can check its struct layout (host function; 0 for other values). */
size_t sa_struct_size(int32_t which);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H_ */
