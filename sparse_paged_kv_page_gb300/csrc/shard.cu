// Sequence sharding: the pages of every request split into contiguous ranges
// held by different shards (devices).
//
// "test_ops_mla_chunked_context.cpp" (vllm.cpp tests), "MergeAttnStates":
// attention over a split of the keys is exact once the partial states are
// merged by their log-sum-exp, lse = log sum_s exp(lse_s), o = sum_s
// exp(lse_s - lse) o_s, an empty part carrying lse = -inf; when every part is
// empty (0/0) the test's reference emits the prefix output, so the merge
// returns part 0's o with lse = -inf (a decode part with no keys holds o = 0). "EntmaxKV" README, "How it works" / "Top-k":
// the selection is the top pages of the whole request with the tail page
// forced, so each shard scores its own pages into its slice of the request's
// score row (the exchange step), one selection is taken over the whole row,
// and each shard attends the selected pages in its range:
//   sa_shard_lengths    the tokens of each request inside a shard's page range
//   sa_shard_selection  the selected pages inside a shard's range, as shard-local
//                       page indices (order kept)
//   sa_merge_states     the partial outputs of the shards merged by log-sum-exp
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

__global__ void shard_lengths_kernel(const int32_t* seq_lens, int B, int ps, int page_lo, int page_hi,
                                     int32_t* out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int64_t L = seq_lens[b];
  const int64_t lo = int64_t(page_lo) * ps, hi = int64_t(page_hi) * ps;
  const int64_t n = L <= lo ? 0 : (L >= hi ? hi - lo : L - lo);
  out[b] = int32_t(n);
}

// one warp per selection unit: ballot compaction keeps the order
__global__ void shard_selection_kernel(const int32_t* sel, const int32_t* cnt, int sel_stride, int units,
                                       int page_lo, int page_hi, int32_t* out, int32_t* out_cnt,
                                       int out_stride, int32_t* status) {
  const int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (u >= units) return;
  int c = cnt[u];
  if (c < 0 || c > sel_stride) {
    if (lane == 0) flag(status, SA_DEV_BAD_COUNT);
    c = c < 0 ? 0 : sel_stride;
  }
  const int32_t* s = sel + int64_t(u) * sel_stride;
  int32_t* o = out + int64_t(u) * out_stride;
  int kept = 0;
  for (int e0 = 0; e0 < c; e0 += 32) {
    const int e = e0 + lane;
    const int p = e < c ? s[e] : -1;
    const bool in = p >= page_lo && p < page_hi;
    const unsigned bal = __ballot_sync(kFull, in);
    const int pos = kept + __popc(bal & ((1u << lane) - 1u));
    if (in) {
      if (pos < out_stride) o[pos] = p - page_lo;
      else flag(status, SA_DEV_OVERFLOW);
    }
    kept += __popc(bal);
  }
  if (lane == 0) out_cnt[u] = min(kept, out_stride);
}

// a part's lse; +inf and NaN count as an empty part, like -inf
__device__ __forceinline__ float part_lse(const float* lse_parts, int64_t i) {
  const float x = lse_parts[i];
  return x < INFINITY ? x : -INFINITY;
}

template <typename T>
__global__ void merge_states_kernel(const uint16_t* o_parts, const float* lse_parts, int S, int rows, int D,
                                    uint16_t* out, float* lse_out) {
  using E = Elem<T>;
  const int r = blockIdx.x;
  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, part_lse(lse_parts, int64_t(s) * rows + r));
  const bool empty = !(m > -INFINITY);
  float l = 0.f;
  if (!empty)
    for (int s = 0; s < S; ++s) l += expf(part_lse(lse_parts, int64_t(s) * rows + r) - m);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    if (empty) {                                // every part empty: the prefix (part 0) output
      out[int64_t(r) * D + d] = o_parts[int64_t(r) * D + d];
      continue;
    }
    float o = 0.f;
    {
      for (int s = 0; s < S; ++s) {
        const float w = expf(part_lse(lse_parts, int64_t(s) * rows + r) - m);   // 0 for an empty part
        if (w > 0.f) o = fmaf(w, E::lo(uint32_t(o_parts[(int64_t(s) * rows + r) * D + d])), o);
      }
      o /= l;
    }
    out[int64_t(r) * D + d] = E::from_f(o);
  }
  if (threadIdx.x == 0 && lse_out) lse_out[r] = empty ? -INFINITY : m + logf(l);
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_shard_lengths(const int32_t* seq_lens, int32_t batch, int32_t page_size,
                                      int32_t page_lo, int32_t page_hi, int32_t* shard_lens,
                                      void* stream) {
  using namespace sa;
  if (!seq_lens || !shard_lens || batch <= 0 || page_size <= 0 || page_lo < 0 || page_hi < page_lo)
    return SA_ERR_INVALID_ARG;
  shard_lengths_kernel<<<(batch + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      seq_lens, batch, page_size, page_lo, page_hi, shard_lens);
  return launch_status();
}

extern "C" sa_status sa_shard_selection(const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_stride,
                                        int32_t num_units, int32_t page_lo, int32_t page_hi,
                                        int32_t* shard_idx, int32_t* shard_cnt, int32_t shard_stride,
                                        int32_t* dev_status, void* stream) {
  using namespace sa;
  if (!sel_idx || !sel_cnt || !shard_idx || !shard_cnt || sel_stride <= 0 || num_units <= 0 ||
      shard_stride <= 0 || page_lo < 0 || page_hi < page_lo)
    return SA_ERR_INVALID_ARG;
  constexpr int kWarps = 8;
  shard_selection_kernel<<<(num_units + kWarps - 1) / kWarps, 32 * kWarps, 0, static_cast<cudaStream_t>(stream)>>>(
      sel_idx, sel_cnt, sel_stride, num_units, page_lo, page_hi, shard_idx, shard_cnt, shard_stride,
      dev_status);
  return launch_status();
}

extern "C" sa_status sa_merge_states(const void* o_parts, const float* lse_parts, int32_t num_shards,
                                     int32_t rows, int32_t head_dim, int32_t dtype, void* out, float* lse,
                                     void* stream) {
  using namespace sa;
  if (!o_parts || !lse_parts || !out || num_shards <= 0 || rows <= 0 || head_dim <= 0)
    return SA_ERR_INVALID_ARG;
  if (dtype != SA_BF16 && dtype != SA_FP16) return SA_ERR_INVALID_ARG;
  const int threads = head_dim >= 128 ? 128 : 64;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* op = static_cast<const uint16_t*>(o_parts);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (dtype == SA_BF16)
    merge_states_kernel<__nv_bfloat16><<<rows, threads, 0, s>>>(op, lse_parts, num_shards, rows, head_dim, o, lse);
  else
    merge_states_kernel<__half><<<rows, threads, 0, s>>>(op, lse_parts, num_shards, rows, head_dim, o, lse);
  return launch_status();
}
