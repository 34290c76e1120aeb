// sa_score_pages: page score of every cached page of every (request, KV head).
//
// "flow: add H2O sparse attention" (vortex_torch PR 6), "Page-level
// variants": average relevance q . mean(k) plus the envelope bound
// sum_d max(q_d max_d, q_d min_d), combined as w_avg * avg + w_peak * peak;
// "EntmaxKV" README, "How it works": pages scored from their statistics
// without touching the cached tokens. The G query heads of a KV head are
// reduced to one ranking by the mean of their scores.
//
// With q+ = max(q, 0), q- = min(q, 0) and max_d >= min_d,
//   max(q max_d, q min_d) = q+ max_d + q- min_d,
// so the group-mean score is
//   S(p) = sum_d [ w_avg qbar_d mean_pd + w_peak (P_d max_pd + N_d min_pd) ]
// with qbar, P, N the group means of q, q+, q-. Each CTA folds the G queries
// of its KV head into those three coefficient vectors once; the page loop is
// then 3 FMAs per element whatever G is, and the kernel is a gather of
// 3 * head_dim * 2 bytes of statistics per page, bounded by HBM bandwidth.
//
// Mapping: a group of head_dim / 8 lanes owns one page; each lane loads the
// 16-byte slice of the page's min, max and mean rows (non-coherent, L1
// bypass), so every 16-lane group reads three contiguous 256-byte rows. Four
// pages per lane group are in flight per iteration.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

struct ScoreArgs {
  const void* meta;
  const void* q;
  const int32_t* bt;
  const int32_t* seq_lens;
  float* scores;
  int32_t* status;
  int H_kv, H_q, G, ps, num_blocks, bt_stride, max_pages;
  float w_avg, w_peak;
};

constexpr int kScoreThreads = 256;
constexpr int kScoreUnroll = 4;
constexpr int kPagesPerCta = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(ScoreArgs a) {
  using E = Elem<T>;
  constexpr int LPP = D / 8;                    // lanes per page
  constexpr int PPP = kScoreThreads / LPP;      // pages per pass
  const int b = blockIdx.z, h = blockIdx.y;
  const int L = a.seq_lens[b];
  int n = (L + a.ps - 1) / a.ps;
  if (n > a.max_pages || n > a.bt_stride) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(a.status, SA_DEV_OVERFLOW);
    n = min(a.max_pages, a.bt_stride);
  }
  const int p_begin = blockIdx.x * kPagesPerCta;
  if (p_begin >= n) return;
  const int p_end = min(n, p_begin + kPagesPerCta);
  const int grp = threadIdx.x / LPP, l = threadIdx.x % LPP;

  // group-mean coefficients of this lane's 8 dimensions
  float ca[8], cp[8], cn[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) ca[e] = cp[e] = cn[e] = 0.f;
  const T* qh = static_cast<const T*>(a.q) + (int64_t(b) * a.H_q + int64_t(h) * a.G) * D + l * 8;
  for (int g = 0; g < a.G; ++g) {
    const uint4 v = *reinterpret_cast<const uint4*>(qh + int64_t(g) * D);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = E::lo(w[e]), x1 = E::hi(w[e]);
      ca[2 * e] += x0; ca[2 * e + 1] += x1;
      cp[2 * e] += fmaxf(x0, 0.f); cp[2 * e + 1] += fmaxf(x1, 0.f);
      cn[2 * e] += fminf(x0, 0.f); cn[2 * e + 1] += fminf(x1, 0.f);
    }
  }
  const float ia = a.w_avg / float(a.G), ip = a.w_peak / float(a.G);
#pragma unroll
  for (int e = 0; e < 8; ++e) { ca[e] *= ia; cp[e] *= ip; cn[e] *= ip; }

  const int32_t* btb = a.bt + int64_t(b) * a.bt_stride;
  float* out = a.scores + (int64_t(b) * a.H_kv + h) * a.max_pages;
  const uint8_t* meta = static_cast<const uint8_t*>(a.meta);
  for (int p0 = p_begin; p0 < p_end; p0 += PPP * kScoreUnroll) {
    uint4 vmn[kScoreUnroll], vmx[kScoreUnroll], vme[kScoreUnroll];
    int state[kScoreUnroll];                     // 0 = no page, 1 = ok, 2 = bad block
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      const int p = p0 + u * PPP + grp;
      state[u] = 0;
      vmn[u] = vmx[u] = vme[u] = make_uint4(0, 0, 0, 0);
      if (p < p_end) {
        const int blk = btb[p];
        if (blk < 0 || blk >= a.num_blocks) {
          state[u] = 2;
        } else {
          state[u] = 1;
          const uint8_t* base =
              meta + ((int64_t(blk) * a.H_kv + h) * 3 * D + l * 8) * int64_t(sizeof(T));
          vmn[u] = ld_nc_v4(base);
          vmx[u] = ld_nc_v4(base + D * sizeof(T));
          vme[u] = ld_nc_v4(base + 2 * D * sizeof(T));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      const uint32_t m0[4] = {vmn[u].x, vmn[u].y, vmn[u].z, vmn[u].w};
      const uint32_t m1[4] = {vmx[u].x, vmx[u].y, vmx[u].z, vmx[u].w};
      const uint32_t m2[4] = {vme[u].x, vme[u].y, vme[u].z, vme[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(ca[2 * e], E::lo(m2[e]), acc);
        acc = fmaf(ca[2 * e + 1], E::hi(m2[e]), acc);
        acc = fmaf(cp[2 * e], E::lo(m1[e]), acc);
        acc = fmaf(cp[2 * e + 1], E::hi(m1[e]), acc);
        acc = fmaf(cn[2 * e], E::lo(m0[e]), acc);
        acc = fmaf(cn[2 * e + 1], E::hi(m0[e]), acc);
      }
#pragma unroll
      for (int o = LPP / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      if (l == 0 && state[u] != 0) {
        const int p = p0 + u * PPP + grp;
        if (state[u] == 2) {
          flag(a.status, SA_DEV_BAD_BLOCK);
          out[p] = __int_as_float(0x7fc00000);
        } else {
          out[p] = acc;
        }
      }
    }
  }
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_score_pages(const sa_cache* cache, const sa_batch* batch, const void* q,
                                    int32_t num_q_heads, float w_avg, float w_peak, float* scores,
                                    int32_t max_pages, int32_t* dev_status, void* stream) {
  using namespace sa;
  sa_status st = check_cache(cache, false, true);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (!q || !scores || max_pages <= 0) return SA_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return SA_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  if (G > 16) return SA_ERR_UNSUPPORTED;
  ScoreArgs a;
  a.meta = cache->meta; a.q = q; a.bt = batch->block_table; a.seq_lens = batch->seq_lens;
  a.scores = scores; a.status = dev_status;
  a.H_kv = cache->num_kv_heads; a.H_q = num_q_heads; a.G = G; a.ps = cache->page_size;
  a.num_blocks = cache->num_blocks; a.bt_stride = batch->bt_stride; a.max_pages = max_pages;
  a.w_avg = w_avg; a.w_peak = w_peak;
  const int cap = max_pages < batch->bt_stride ? max_pages : batch->bt_stride;
  dim3 grid(unsigned((cap + kPagesPerCta - 1) / kPagesPerCta), unsigned(a.H_kv),
            unsigned(batch->batch));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = cache->dtype == SA_BF16;
  if (cache->head_dim == 128) {
    if (bf) score_kernel<__nv_bfloat16, 128><<<grid, kScoreThreads, 0, s>>>(a);
    else score_kernel<__half, 128><<<grid, kScoreThreads, 0, s>>>(a);
  } else {
    if (bf) score_kernel<__nv_bfloat16, 64><<<grid, kScoreThreads, 0, s>>>(a);
    else score_kernel<__half, 64><<<grid, kScoreThreads, 0, s>>>(a);
  }
  return launch_status();
}
