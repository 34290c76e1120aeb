// sa_decode_step: one page-level decode step (append, score, select, sparse
// decode) enqueued as one chain of programmatically dependent launches.
//
// The order of the step is the one of "flow: add H2O sparse attention
// (page-level and token-level, MHA + GQA)", section "Page-level variants"
// (statistics refreshed on append, pages scored from them, top-k, attention
// over the chosen pages), and of the EntmaxKV README, "How it works".
//
// Overlap. With one new token per request the append writes only the tail
// page: either the old tail (which stays the tail) or a fresh page past the
// old length. Every other page's statistics are final before the step starts,
// so the scorer can run on the lengths it reads at entry while the append runs
// beside it; the tail is always selected, so its score does not influence the
// selection. With more new tokens a page can stop being the tail inside the
// step, and the append runs first.
#include "host.h"

extern "C" sa_status sa_decode_step(const sa_cache* cache, const sa_batch* batch, const void* k_new,
                                    const void* v_new, const int32_t* new_cu,
                                    int32_t max_new_per_req, const void* q, int32_t num_q_heads,
                                    float w_avg, float w_peak, float* scores, int32_t max_pages,
                                    int32_t topk, int32_t n_bos, int32_t n_eos, int32_t* sel_idx,
                                    int32_t* sel_cnt, float scale,
                                    void* out, float* lse, void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, void* stream) {
  using namespace sa;
  // every argument of the four stages is checked before anything is launched
  sa_status st = check_cache(cache, true, true);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  const bool append = k_new != nullptr && max_new_per_req > 0;
  if (append && (!v_new || !new_cu)) return SA_ERR_INVALID_ARG;
  if (!q || !scores || !sel_idx || !sel_cnt || !out || max_pages <= 0 || topk <= 0 ||
      max_new_per_req < 0 || n_bos < 0 || n_eos < 1 || n_bos + n_eos > topk)
    return SA_ERR_INVALID_ARG;
  if (!aligned16(q)) return SA_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return SA_ERR_INVALID_ARG;
  if (num_q_heads / cache->num_kv_heads > 16) return SA_ERR_UNSUPPORTED;
  if (batch->batch > 1024 || max_pages > 45056) return SA_ERR_UNSUPPORTED;
  const size_t need = sa_decode_workspace_size(batch->batch, cache->num_kv_heads, num_q_heads,
                                               cache->head_dim, cache->page_size, topk);
  if (need == 0) return SA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need) return SA_ERR_WORKSPACE;

  const bool overlap = append && max_new_per_req == 1;
  if (append && !overlap) {
    st = append_impl(cache, batch, k_new, v_new, new_cu, max_new_per_req, nullptr, nullptr, nullptr,
                     0, dev_status, stream, false);
    if (st != SA_OK) return st;
  }
  st = score_impl(cache, batch, q, num_q_heads, w_avg, w_peak, scores, max_pages, dev_status, stream,
                  false);
  if (st != SA_OK) return st;
  if (overlap) {
    st = append_impl(cache, batch, k_new, v_new, new_cu, 1, nullptr, nullptr, nullptr, 0, dev_status,
                     stream, true);
    if (st != SA_OK) return st;
  }
  st = select_impl(scores, max_pages, batch, cache->page_size, cache->num_kv_heads, topk, n_bos,
                   n_eos, sel_idx, sel_cnt, dev_status, stream, true);
  if (st != SA_OK) return st;
  return decode_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, topk, scale, out, lse, nullptr, 0,
                     workspace, workspace_bytes, dev_status, stream, true, true, false, false);
}
