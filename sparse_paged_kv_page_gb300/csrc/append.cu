// sa_append_kv: write new keys / values into the paged pools and recompute
// the element-wise statistics (k_min, k_max, k_mean, and k_std where the cache
// keeps it) of every page touched.
//
// "flow: add H2O sparse attention" (vortex_torch PR 6), "Page-level variants"
// and "Token-level variants" point 2: the statistics are overwriting
// reductions over the written page, and the H2O score slots written in the
// step are reset to zero because recycled pool pages keep stale contents.
// "EntmaxKV" README, "How it works": per-page key statistics refreshed on
// append (min / max for top-k, mean / std for the Gaussian strategy).
//
// One CTA per (touched page, request); thread (h, c) owns the column pair
// [2c, 2c+1] of KV head h and loads all of the page's rows before using any,
// taking new rows from the input and old ones from the pool, so no other
// CTA's writes are read and a page costs one memory round trip per 16 rows.
// Slots past the page's new fill are stale and never touched.
//
// k_mean is the float64 mean rounded once to the cache dtype. GB300's float64
// rate is low, so the kernel computes it in float32 and proves the result
// exact: each running sum carries a TwoSum error term (zero => the float32
// sum is the exact sum S); S / f in float32 is correctly rounded, and
// rounding it to the dtype equals rounding S / f itself unless the float32
// quotient lands exactly on a dtype midpoint, which is then settled by the
// exact product midpoint * f against S. Columns where any of this does not
// hold (an inexact running sum, float32 underflow, fp16 subnormals) recompute
// in float64 from the pool.
//
// When every request touches at most two pages (decode), one CTA per request
// handles its pages and then advances the request's length itself; otherwise
// a second one-block kernel advances the lengths after all CTAs have read them.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

struct AppendArgs {
  void* k;
  void* v;
  void* meta;
  void* kstd;
  const void* k_new;
  const void* v_new;
  const int32_t* new_cu;
  const int32_t* bt;
  int32_t* seq_lens;
  uint16_t* hh;
  int32_t* ret_pos;
  int32_t* ret_cnt;
  int32_t* status;
  int H, D, ps, num_blocks, bt_stride, max_new, ret_cap;
};

constexpr int kAppendThreads = 512;   // prefill path
constexpr int kFusedThreads = 128;    // decode path: small enough to run beside the page scorer
constexpr int kRowBatch = 16;     // rows of a page loaded per batch (independent loads)

// exact float32 sum step: s += x, clears `exact` if the addition rounded
__device__ __forceinline__ void two_sum(float& s, float x, bool& exact) {
  const float t = s + x;
  const float bb = t - s;
  const float err = (s - (t - bb)) + (x - bb);
  exact &= (err == 0.f);
  s = t;
}

// Round S / f (S exact) once to the element type; false if float32 cannot decide.
template <typename T>
__device__ __forceinline__ bool mean_f32(float S, int f, uint16_t& out) {
  using E = Elem<T>;
  const float aS = fabsf(S);
  if (S == 0.f) { out = E::from_f(S); return true; }
  if (!(aS >= 0x1p-100f)) return false;                       // float32 underflow risk
  if ((f & (f - 1)) == 0) {                                    // power of two: exact scaling
    const float q = S * (1.0f / float(f));
    if (E::midpoint(q) < 0) return false;
    out = E::from_f(q);
    return true;
  }
  const float q = S / float(f);                                // correctly rounded
  const int mid = E::midpoint(q);
  if (mid < 0) return false;
  if (mid == 0) { out = E::from_f(q); return true; }
  const float prod = q * float(f);                             // exact: few significant bits
  if (S == prod) { out = E::from_f(q); return true; }          // a true tie: to even
  const uint16_t lo = E::from_f_rz(fabsf(q));                  // smaller-magnitude neighbour
  const uint16_t mag = fabsf(S) > fabsf(prod) ? uint16_t(lo + 1) : lo;
  out = uint16_t(mag | (S < 0.f ? 0x8000u : 0u));
  return true;
}

// k_std of one column over its f rows: the population std sqrt((1/f) sum
// (x - mean)^2) around the exact mean, rounded once to the element type.
// float32 two-pass: with m the float32 mean (error dm <= (f + 1) eps sum|x| / f)
// the computed sum of squared deviations q differs from the true one by at
// most f dm^2 (the centre's error enters squared, the deviations summing to
// zero) plus (f + 3) eps q of rounding, so the std's relative error is below
// half that (+ eps). The float32 result is kept when every value within twice
// that bound rounds to the same element; otherwise float64 decides. x: the
// column's values (half kHi of each word), f <= kRowBatch of them.
template <typename T, bool kHi>
__device__ __forceinline__ uint16_t std_column(const uint32_t (&w)[kRowBatch], int fill) {
  using E = Elem<T>;
  constexpr float eps = 0x1p-24f;
  float sum = 0.f, sabs = 0.f, xmin = INFINITY, xmax = -INFINITY;
#pragma unroll
  for (int s = 0; s < kRowBatch; ++s) {
    if (s < fill) {
      const float x = kHi ? E::hi(w[s]) : E::lo(w[s]);
      sum += x;
      sabs += fabsf(x);
      xmin = fminf(xmin, x);
      xmax = fmaxf(xmax, x);
    }
  }
  if (xmin == xmax) return E::from_f(0.f);                 // every row equal
  const float f = float(fill);
  const float m = sum / f;
  float q = 0.f;
#pragma unroll
  for (int s = 0; s < kRowBatch; ++s) {
    if (s < fill) {
      const float d = (kHi ? E::hi(w[s]) : E::lo(w[s])) - m;
      q = fmaf(d, d, q);
    }
  }
  const float dm = (f + 1.f) * eps * sabs / f;
  const float rel = 0.5f * (f * dm * dm / q + (f + 3.f) * eps) + eps;
  const float sd = sqrtf(q / f);
  if (q > 0x1p-100f && rel < 0x1p-12f) {
    const uint16_t lo = E::from_f(sd * (1.f - 2.f * rel)), hi = E::from_f(sd * (1.f + 2.f * rel));
    if (lo == hi) return lo;
  }
  double s64 = 0.0;                                        // undecided: float64
#pragma unroll
  for (int s = 0; s < kRowBatch; ++s)
    if (s < fill) s64 += double(kHi ? E::hi(w[s]) : E::lo(w[s]));
  const double m64 = s64 / double(fill);
  double q64 = 0.0;
#pragma unroll
  for (int s = 0; s < kRowBatch; ++s) {
    if (s < fill) {
      const double d = double(kHi ? E::hi(w[s]) : E::lo(w[s])) - m64;
      q64 = fma(d, d, q64);
    }
  }
  return E::from_f64(sqrt(q64 / double(fill)));
}

// float64 k_std of one column over more rows than one batch (pages above 16 tokens)
template <typename T, bool kHi>
__device__ uint16_t std_column_long(const uint32_t* rows, int C, int fill) {
  using E = Elem<T>;
  double s64 = 0.0;
  for (int s = 0; s < fill; ++s) s64 += double(kHi ? E::hi(rows[int64_t(s) * C]) : E::lo(rows[int64_t(s) * C]));
  const double m64 = s64 / double(fill);
  double q64 = 0.0;
  for (int s = 0; s < fill; ++s) {
    const double d = double(kHi ? E::hi(rows[int64_t(s) * C]) : E::lo(rows[int64_t(s) * C])) - m64;
    q64 = fma(d, d, q64);
  }
  return E::from_f64(sqrt(q64 / double(fill)));
}

// k_std of the column pair [2c, 2c+1] of (block, head); the f rows, new ones
// included, are this thread's own pool writes or untouched. Only for caches
// that keep k_std; kept out of line so the common path keeps its registers.
template <typename T>
__device__ __noinline__ void page_std_pair(const AppendArgs& a, const uint32_t* kp, int64_t tile,
                                           int fill, int blk, int h, int c) {
  const int C = a.D / 2;
  const uint32_t* rows = kp + tile * C + c;
  uint16_t v0, v1;
  if (fill <= kRowBatch) {
    uint32_t w[kRowBatch];
#pragma unroll
    for (int s = 0; s < kRowBatch; ++s) w[s] = s < fill ? rows[int64_t(s) * C] : 0u;   // one batch of loads
    v0 = std_column<T, false>(w, fill);
    v1 = std_column<T, true>(w, fill);
  } else {
    v0 = std_column_long<T, false>(rows, C, fill);
    v1 = std_column_long<T, true>(rows, C, fill);
  }
  static_cast<uint32_t*>(a.kstd)[(int64_t(blk) * a.H + h) * C + c] = uint32_t(v0) | (uint32_t(v1) << 16);
}

// Recompute statistics of page p of request b (all heads) and write the new rows.
// Thread (h, c) owns the column pair [2c, 2c+1] of KV head h (NT threads loop).
template <typename T, int NT, bool kStd>
__device__ __forceinline__ void refresh_page(const AppendArgs& a, int b, int p, int L_old, int L_new,
                                             int row0) {
  using E = Elem<T>;
  const int ps = a.ps, H = a.H, D = a.D;
  const int blk = a.bt[int64_t(b) * a.bt_stride + p];
  if (blk < 0 || blk >= a.num_blocks) {
    if (threadIdx.x == 0) flag(a.status, SA_DEV_BAD_BLOCK);
    return;
  }
  const int page_start = p * ps;
  const int fill = min(ps, L_new - page_start);          // valid tokens after the append
  const int s_new = max(0, L_old - page_start);          // first slot written here
  const int C = D / 2;                                    // column pairs per row
  const uint32_t* kn = static_cast<const uint32_t*>(a.k_new);
  const uint32_t* vn = static_cast<const uint32_t*>(a.v_new);
  uint32_t* kp = static_cast<uint32_t*>(a.k);
  uint32_t* vp = static_cast<uint32_t*>(a.v);

  for (int idx = threadIdx.x; idx < H * C; idx += NT) {
    const int h = idx / C, c = idx % C;
    const int64_t tile = (int64_t(blk) * H + h) * ps;    // first row of this (block, head)
    float mn0 = INFINITY, mn1 = INFINITY, mx0 = -INFINITY, mx1 = -INFINITY, sm0 = 0.f, sm1 = 0.f;
    bool ex0 = true, ex1 = true;
    uint32_t r[kRowBatch];
    for (int s0 = 0; s0 < fill; s0 += kRowBatch) {
#pragma unroll
      for (int j = 0; j < kRowBatch; ++j) {
        const int s = s0 + j;
        r[j] = 0u;
        if (s < fill) {
          if (s >= s_new) r[j] = kn[(int64_t(row0 + page_start + s - L_old) * H + h) * C + c];
          else r[j] = kp[(tile + s) * C + c];
        }
      }
#pragma unroll
      for (int j = 0; j < kRowBatch; ++j) {
        if (s0 + j < fill) {
          const float x0 = E::lo(r[j]), x1 = E::hi(r[j]);
          mn0 = fminf(mn0, x0); mn1 = fminf(mn1, x1);
          mx0 = fmaxf(mx0, x0); mx1 = fmaxf(mx1, x1);
          two_sum(sm0, x0, ex0);
          two_sum(sm1, x1, ex1);
        }
      }
#pragma unroll
      for (int j = 0; j < kRowBatch; ++j) {                // the new rows go to the pool
        const int s = s0 + j;
        if (s < fill && s >= s_new) {
          const int64_t src = (int64_t(row0 + page_start + s - L_old) * H + h) * C + c;
          kp[(tile + s) * C + c] = r[j];
          vp[(tile + s) * C + c] = vn[src];
        }
      }
    }
    if (!a.meta) continue;
    uint16_t me0 = 0, me1 = 0;
    ex0 = ex0 && mean_f32<T>(sm0, fill, me0);
    ex1 = ex1 && mean_f32<T>(sm1, fill, me1);
    if (!ex0 || !ex1) {                                   // rare: float64
      double d0 = 0.0, d1 = 0.0;
      if (fill <= kRowBatch) {
#pragma unroll
        for (int j = 0; j < kRowBatch; ++j)
          if (j < fill) { d0 += double(E::lo(r[j])); d1 += double(E::hi(r[j])); }
      } else {
        for (int s = 0; s < fill; ++s) {
          const uint32_t x = kp[(tile + s) * C + c];
          d0 += double(E::lo(x));
          d1 += double(E::hi(x));
        }
      }
      if (!ex0) me0 = E::from_f64(d0 / double(fill));
      if (!ex1) me1 = E::from_f64(d1 / double(fill));
    }
    uint32_t* m = static_cast<uint32_t*>(a.meta) + (int64_t(blk) * H + h) * 3 * C + c;
    m[0] = E::pack(mn0, mn1);                             // exact: values are already dtype
    m[C] = E::pack(mx0, mx1);
    m[2 * C] = uint32_t(me0) | (uint32_t(me1) << 16);
    if constexpr (kStd) {
      if (fill <= kRowBatch) {                            // the rows are still in registers
        const uint16_t v0 = std_column<T, false>(r, fill), v1 = std_column<T, true>(r, fill);
        static_cast<uint32_t*>(a.kstd)[(int64_t(blk) * H + h) * C + c] = uint32_t(v0) | (uint32_t(v1) << 16);
      } else {
        page_std_pair<T>(a, kp, tile, fill, blk, h, c);
      }
    }
  }
  // H2O slots of the written tokens start at zero
  if (a.hh) {
    for (int idx = threadIdx.x; idx < (fill - s_new) * H; idx += NT) {
      const int s = s_new + idx / H, h = idx % H;
      a.hh[(int64_t(blk) * ps + s) * H + h] = 0;
    }
  }
  // token-level retained lists: append the new positions, ascending
  if (a.ret_pos) {
    for (int idx = threadIdx.x; idx < (fill - s_new) * H; idx += NT) {
      const int s = s_new + idx / H, h = idx % H;
      const int pos = page_start + s;
      const int cpos = a.ret_cnt[b * H + h] + (pos - L_old);
      if (cpos < 0 || cpos >= a.ret_cap) {
        flag(a.status, SA_DEV_OVERFLOW);
        continue;
      }
      a.ret_pos[(int64_t(b) * H + h) * a.ret_cap + cpos] = pos;
    }
  }
}

// Clamp request b's new-token count; returns false if nothing is appended.
__device__ __forceinline__ bool plan(const AppendArgs& a, int b, bool report, int& L_old, int& n,
                                     int& row0) {
  L_old = a.seq_lens[b];
  row0 = a.new_cu[b];
  n = a.new_cu[b + 1] - row0;
  if (n > a.max_new) {
    if (report) flag(a.status, SA_DEV_OVERFLOW);
    n = a.max_new;
  }
  const int64_t cap_tok = int64_t(a.bt_stride) * a.ps;
  if (L_old < 0 || L_old > cap_tok) {
    if (report) flag(a.status, SA_DEV_OVERFLOW);
    return false;
  }
  if (L_old + int64_t(n) > cap_tok) {
    if (report) flag(a.status, SA_DEV_OVERFLOW);
    n = int(cap_tok - L_old);
  }
  return n > 0;
}

// Grid (touched pages, B); lengths advanced by advance_kernel afterwards.
template <typename T, bool kStd>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(AppendArgs a) {
  const int b = blockIdx.y, i = blockIdx.x;
  int L_old, n, row0;
  if (!plan(a, b, i == 0 && threadIdx.x == 0, L_old, n, row0)) return;
  const int p = L_old / a.ps + i;
  if (p > (L_old + n - 1) / a.ps) return;
  refresh_page<T, kAppendThreads, kStd>(a, b, p, L_old, L_old + n, row0);
}

// Grid (B): a request's (at most two) pages, then its length, in one CTA.
// NT = kFusedThreads when launched beside the page scorer: at most 128
// registers a thread, and with the scorer's two CTAs resident the
// sub-partitions holding three of its warps have exactly one 128-register
// warp's worth of registers left. A plain launch takes NT = kAppendThreads,
// one (head, column pair) a thread at 8 KV heads of 128 dimensions.
template <typename T, bool kStd, int NT>
__global__ void __launch_bounds__(NT, 512 / NT) append_fused_kernel(AppendArgs a) {
  const int b = blockIdx.x;
  int L_old, n, row0;
  const bool any = plan(a, b, threadIdx.x == 0, L_old, n, row0);
  if (any)
    for (int p = L_old / a.ps; p <= (L_old + n - 1) / a.ps; ++p)
      refresh_page<T, NT, kStd>(a, b, p, L_old, L_old + n, row0);
  __syncthreads();                                          // every read of the old length is done
  if (any) {
    for (int h = threadIdx.x; h < a.H && a.ret_cnt; h += NT) {
      const int c = a.ret_cnt[b * a.H + h] + n;
      a.ret_cnt[b * a.H + h] = min(max(c, 0), a.ret_cap);
    }
    if (threadIdx.x == 0) a.seq_lens[b] = L_old + n;
  }
  // Launched programmatically beside the page scorer (which has read the old
  // lengths before letting this kernel start), it finishes only after the
  // scorer, so whatever follows in the stream sees both.
  pdl_wait();
}

// Advances lengths (and retained counts) after the append kernel has read them.
__global__ void advance_kernel(int32_t* seq_lens, const int32_t* new_cu, int32_t* ret_cnt, int B,
                               int H, int max_new, int64_t cap_tok, int ret_cap) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int L = seq_lens[b];
    if (L < 0 || L > cap_tok) continue;
    int n = new_cu[b + 1] - new_cu[b];
    n = max(0, min(n, max_new));
    const int64_t Ln = min(int64_t(L) + n, cap_tok);
    seq_lens[b] = int32_t(Ln);
    if (ret_cnt) {
      const int add = int(Ln - L);
      for (int h = 0; h < H; ++h) {
        const int c = ret_cnt[b * H + h] + add;
        ret_cnt[b * H + h] = min(max(c, 0), ret_cap);
      }
    }
  }
}

}  // namespace
}  // namespace sa

sa_status sa::append_impl(const sa_cache* cache, const sa_batch* batch, const void* k_new,
                         const void* v_new, const int32_t* new_cu, int32_t max_new_per_req, void* hh,
                         int32_t* ret_pos, int32_t* ret_cnt, int32_t ret_cap, int32_t* dev_status,
                         void* stream, bool pdl) {
  using namespace sa;
  sa_status st = check_cache(cache, true, false);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (!k_new || !v_new || !new_cu || max_new_per_req < 0) return SA_ERR_INVALID_ARG;
  if ((ret_pos == nullptr) != (ret_cnt == nullptr)) return SA_ERR_INVALID_ARG;
  if (ret_pos && ret_cap <= 0) return SA_ERR_INVALID_ARG;
  if (max_new_per_req == 0) return SA_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AppendArgs a;
  a.k = cache->k; a.v = cache->v; a.meta = cache->meta; a.kstd = cache->meta ? cache->kstd : nullptr;
  a.k_new = k_new; a.v_new = v_new; a.new_cu = new_cu;
  a.bt = batch->block_table; a.seq_lens = batch->seq_lens;
  a.hh = static_cast<uint16_t*>(hh); a.ret_pos = ret_pos; a.ret_cnt = ret_cnt;
  a.status = dev_status;
  a.H = cache->num_kv_heads; a.D = cache->head_dim; a.ps = cache->page_size;
  a.num_blocks = cache->num_blocks; a.bt_stride = batch->bt_stride;
  a.max_new = max_new_per_req; a.ret_cap = ret_pos ? ret_cap : 0;
  const bool bf = cache->dtype == SA_BF16;
  if (max_new_per_req <= a.ps) {                            // touches at most two pages per request
    static int g_fused_attr[8][64];
    auto kern = pdl ? (bf ? (a.kstd ? append_fused_kernel<__nv_bfloat16, true, kFusedThreads>
                                    : append_fused_kernel<__nv_bfloat16, false, kFusedThreads>)
                          : (a.kstd ? append_fused_kernel<__half, true, kFusedThreads>
                                    : append_fused_kernel<__half, false, kFusedThreads>))
                    : (bf ? (a.kstd ? append_fused_kernel<__nv_bfloat16, true, kAppendThreads>
                                    : append_fused_kernel<__nv_bfloat16, false, kAppendThreads>)
                          : (a.kstd ? append_fused_kernel<__half, true, kAppendThreads>
                                    : append_fused_kernel<__half, false, kAppendThreads>));
    if (!ensure_smem(kern, 0, g_fused_attr[(pdl ? 0 : 4) + (bf ? 0 : 2) + (a.kstd ? 1 : 0)])) return SA_ERR_CUDA;
    const cudaError_t e =
        launch_ex(kern, dim3(batch->batch), dim3(pdl ? kFusedThreads : kAppendThreads), 0, s, pdl, 1, a);
    return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
  }
  const int64_t pages = (int64_t(max_new_per_req) + a.ps - 1) / a.ps + 1;
  if (pages > 0x7fffffff) return SA_ERR_INVALID_ARG;
  dim3 grid(unsigned(pages), unsigned(batch->batch));
  auto kern = bf ? (a.kstd ? append_kernel<__nv_bfloat16, true> : append_kernel<__nv_bfloat16, false>)
                 : (a.kstd ? append_kernel<__half, true> : append_kernel<__half, false>);
  kern<<<grid, kAppendThreads, 0, s>>>(a);
  if ((st = launch_status()) != SA_OK) return st;
  advance_kernel<<<1, 256, 0, s>>>(batch->seq_lens, new_cu, ret_cnt, batch->batch, a.H,
                                   max_new_per_req, int64_t(batch->bt_stride) * a.ps, a.ret_cap);
  return launch_status();
}

extern "C" sa_status sa_append_kv(const sa_cache* cache, const sa_batch* batch, const void* k_new,
                                  const void* v_new, const int32_t* new_cu, int32_t max_new_per_req,
                                  void* hh, int32_t* ret_pos, int32_t* ret_cnt, int32_t ret_cap,
                                  int32_t* dev_status, void* stream) {
  return sa::append_impl(cache, batch, k_new, v_new, new_cu, max_new_per_req, hh, ret_pos, ret_cnt,
                         ret_cap, dev_status, stream, false);
}
