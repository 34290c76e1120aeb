// sa_select_topk: the pages each (request, KV head) attends.
//
// "EntmaxKV" README, "How it works", "Top-k": keep topk pages, the budget
// counting pages and including the always-attended tail page. With n pages:
// n <= topk keeps all; otherwise the tail n-1 plus the topk-1 best of pages
// 0..n-2 by (score descending, index ascending); -0 == +0; NaN ranks last.
// "flow: add H2O sparse attention" (vortex_torch PR 6), the follow-up comment:
// page_reserved_bos leading and page_reserved_eos trailing pages are kept
// unconditionally and top-k ranks only the window between them
// (sa_select_topk_reserved; the reserved pages count against the budget, so
// n_bos = 0, n_eos = 1 is the rule above).
//
// One 1024-thread CTA per (KV head, request). Scores become order-preserving
// 32-bit keys in shared memory; a most-significant-digit radix select
// (12-, 12- and 8-bit digits, early exit once a digit bin is taken whole) finds the
// key K of the (topk-1)-th best candidate and how many candidates equal to K
// to keep; those are the lowest-indexed ones. Warp ballots over contiguous
// segments, with one exchange of per-warp counts, then give each kept page its
// slot in page order, so the output is ascending without sorting and the
// result is deterministic.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

#ifndef SA_SELECT_THREADS
#define SA_SELECT_THREADS 1024
#endif
constexpr int kSelThreads = SA_SELECT_THREADS;
constexpr int kBpt = 4096 / kSelThreads;   // histogram bins owned per thread in the digit search
constexpr int kWarps = kSelThreads / 32;
constexpr int kFirst = 9;                  // candidates a thread loads with the length
static_assert(kSelThreads == 1024, "the digit search maps 4096 bins and 32 warps onto the block");
constexpr int kSelMaxPages = 45056;      // keys in shared memory next to two 16 KB histograms

struct SelArgs {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* sel_idx;
  int32_t* sel_cnt;
  int32_t* status;
  int H, ps, max_pages, topk;
  int n_bos, n_eos;      // reserved leading / trailing pages (n_eos >= 1: the tail)
};

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[2][4096];                  // digit histograms, alternating per pass
  __shared__ int s_wt[kWarps], s_gt[kWarps], s_eq[kWarps];
  __shared__ int s_digit, s_above, s_whole;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int unit = b * a.H + h;
  pdl_wait();                                  // scores and lengths of this step are final
  pdl_trigger();                               // the decode may start its prologue
  // Candidate i is page n_bos + i. The first kFirst * kSelThreads
  // candidates' scores are loaded together with the length (the row holds
  // max_pages entries; entries past the length are ignored): 9 a thread, so
  // the 8193 candidates of a 131072-token request need one round trip.
  const int bos = a.n_bos, eos = a.n_eos;
  const float* sc = a.scores + int64_t(unit) * a.max_pages + bos;
  float v0[kFirst];
#pragma unroll
  for (int u = 0; u < kFirst; ++u) {
    const int i = u * kSelThreads + tid;
    v0[u] = bos + i < a.max_pages ? sc[i] : 0.f;
  }
  const int L = a.seq_lens[b];
  int n = L > 0 ? (L + a.ps - 1) / a.ps : 0;
  if (n > a.max_pages) {
    if (tid == 0) flag(a.status, SA_DEV_OVERFLOW);
    n = a.max_pages;
  }
  int32_t* out = a.sel_idx + int64_t(unit) * a.topk;
  if (n <= a.topk) {
    for (int i = tid; i < n; i += kSelThreads) out[i] = i;
    if (tid == 0) a.sel_cnt[unit] = n;
    return;
  }
  // the reserved pages: 0 .. bos-1 first, n-eos .. n-1 last (the tail among them)
  const int kprime = a.topk - bos - eos;         // best candidates besides the reserved pages
  const int nc = n - bos - eos;                  // candidates: pages bos .. n-eos-1
  for (int j = tid; j < bos; j += kSelThreads) out[j] = j;
  for (int j = tid; j < eos; j += kSelThreads) out[bos + kprime + j] = n - eos + j;
  if (tid == 0) a.sel_cnt[unit] = a.topk;
  if (kprime == 0) return;
  for (int i = tid; i < 2 * 4096; i += kSelThreads) (&hist[0][0])[i] = 0;
  __syncthreads();
  // keys to shared memory; the first digit's histogram straight from registers
#pragma unroll
  for (int u = 0; u < kFirst; ++u) {
    const int i = u * kSelThreads + tid;
    if (i < nc) {
      const uint32_t k = f32_key(v0[u]);
      keys[i] = k;
      atomicAdd(&hist[0][k >> 20], 1);
    }
  }
  for (int i0 = kFirst * kSelThreads; i0 < nc; i0 += 8 * kSelThreads) {   // long rows
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelThreads + tid;
      v[u] = i < nc ? sc[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelThreads + tid;
      if (i < nc) {
        const uint32_t k = f32_key(v[u]);
        keys[i] = k;
        atomicAdd(&hist[0][k >> 20], 1);
      }
    }
  }

  // Radix select from the most significant digit: 12, 12 and 8 bits. (The top
  // byte of a float key is the sign and high exponent bits -- a 12-bit first
  // digit also takes three mantissa bits, so the first pass already splits
  // typical score distributions into many bins.) Warp w owns a contiguous run
  // of bins from the top, lane l kBpt of them, so the bin holding the
  // remaining-th largest key is found with two barriers per digit.
  uint32_t prefix = 0, mask = 0;
  int remaining = kprime;                        // still to take among keys matching prefix
  for (int pass = 0; pass < 3; ++pass) {
    const int width = pass < 2 ? 12 : 8;
    const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
    const int nbins = 1 << width;
    int* hp = hist[pass & 1];
    if (pass > 0) {
      for (int i = tid; i < nc; i += kSelThreads) {
        const uint32_t k = keys[i];
        if ((k & mask) == prefix) atomicAdd(&hp[(k >> shift) & uint32_t(nbins - 1)], 1);
      }
    }
    __syncthreads();                             // histogram complete
    const int bpl = nbins / kSelThreads;         // bins per lane: 4 (12-bit) or 0 (8-bit)
    int c[kBpt], sum = 0, top;
    if (bpl) {
      top = nbins - 1 - kBpt * tid;              // lane's bins top, top-1, ..., top-kBpt+1
#pragma unroll
      for (int j = 0; j < kBpt; ++j) { c[j] = hp[top - j]; sum += c[j]; }
    } else {                                     // 256 bins: one per thread of warps 0..7
      top = nbins - 1 - tid;
#pragma unroll
      for (int j = 0; j < kBpt; ++j) c[j] = 0;
      if (tid < nbins) { c[0] = hp[top]; sum = c[0]; }
    }
    int incl = sum;                              // inclusive scan over the warp's lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_wt[warp] = incl;
    __syncthreads();                             // warp totals published, histogram read
    if (pass == 0)                               // the third digit reuses this buffer
      for (int i = tid; i < 256; i += kSelThreads) hist[0][i] = 0;
    int wt = lane < kWarps ? s_wt[lane] : 0;
    int wincl = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, wincl, o);
      if (lane >= o) wincl += y;
    }
    const int wbefore = __shfl_sync(kFull, wincl - wt, warp);
    int run = wbefore + incl - sum;              // keys in bins above this lane's first bin
#pragma unroll
    for (int j = 0; j < kBpt; ++j) {
      if (run < remaining && remaining <= run + c[j]) {
        s_digit = top - j;
        s_above = run;
        s_whole = (run + c[j] == remaining);
      }
      run += c[j];
    }
    __syncthreads();                             // digit published
    const int d = s_digit;
    remaining -= s_above;
    prefix |= uint32_t(d) << shift;
    mask |= uint32_t(nbins - 1) << shift;
    if (s_whole) break;
  }

  // keep: (key & mask) > prefix, or == prefix among the first `remaining` in
  // page order. Warp w walks a contiguous segment in rounds of 32; ballots
  // count and rank within a round, one barrier shares the per-warp counts.
  const int seg = (((nc + kWarps - 1) / kWarps) + 31) & ~31;
  const int s0 = warp * seg, s1 = min(nc, s0 + seg);
  const uint32_t lt = (1u << lane) - 1u;
  int gt = 0, eq = 0;
  for (int base = s0; base < s1; base += 32) {
    const int i = base + lane;
    const uint32_t k = i < s1 ? keys[i] & mask : 0u;
    gt += __popc(__ballot_sync(kFull, i < s1 && k > prefix));
    eq += __popc(__ballot_sync(kFull, i < s1 && k == prefix));
  }
  if (lane == 0) { s_gt[warp] = gt; s_eq[warp] = eq; }
  __syncthreads();
  int g = lane < kWarps ? s_gt[lane] : 0, e = lane < kWarps ? s_eq[lane] : 0;
  const int g_own = g, e_own = e;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yg = __shfl_up_sync(kFull, g, o), ye = __shfl_up_sync(kFull, e, o);
    if (lane >= o) { g += yg; e += ye; }
  }
  const int gt_before = __shfl_sync(kFull, g - g_own, warp);
  int eq_run = __shfl_sync(kFull, e - e_own, warp);
  int take_run = gt_before + min(eq_run, remaining);
  for (int base = s0; base < s1; base += 32) {
    const int i = base + lane;
    const uint32_t k = i < s1 ? keys[i] & mask : 0u;
    const bool is_gt = i < s1 && k > prefix, is_eq = i < s1 && k == prefix;
    const uint32_t meq = __ballot_sync(kFull, is_eq);
    const bool take = is_gt || (is_eq && eq_run + __popc(meq & lt) < remaining);
    const uint32_t mt = __ballot_sync(kFull, take);
    const int pos = take_run + __popc(mt & lt);
    if (take && pos < kprime) out[bos + pos] = bos + i;
    eq_run += __popc(meq);
    take_run += __popc(mt);
  }
}

int g_sel_smem[64];

}  // namespace
}  // namespace sa

sa_status sa::select_impl(const float* scores, int32_t max_pages, const sa_batch* batch,
                         int32_t page_size, int32_t num_kv_heads, int32_t topk, int32_t n_bos,
                         int32_t n_eos, int32_t* sel_idx, int32_t* sel_cnt, int32_t* dev_status,
                         void* stream, bool pdl) {
  using namespace sa;
  sa_status st = check_batch(batch);
  if (st != SA_OK) return st;
  if (!scores || !sel_idx || !sel_cnt || max_pages <= 0 || num_kv_heads <= 0 || topk <= 0)
    return SA_ERR_INVALID_ARG;
  if (!is_pow2(page_size) || page_size > 128) return SA_ERR_UNSUPPORTED;
  if (max_pages > kSelMaxPages) return SA_ERR_UNSUPPORTED;
  if (n_bos < 0 || n_eos < 1 || n_bos + n_eos > topk) return SA_ERR_INVALID_ARG;
  SelArgs a;
  a.scores = scores; a.seq_lens = batch->seq_lens; a.sel_idx = sel_idx; a.sel_cnt = sel_cnt;
  a.status = dev_status; a.H = num_kv_heads; a.ps = page_size; a.max_pages = max_pages;
  a.topk = topk; a.n_bos = n_bos; a.n_eos = n_eos;
  const int smem = max_pages * int(sizeof(uint32_t));
  // static shared memory (the 16 KB histogram) plus the keys may pass the 48 KB default
  if (!ensure_smem(select_kernel, smem, g_sel_smem)) return SA_ERR_CUDA;
  dim3 grid(unsigned(num_kv_heads), unsigned(batch->batch));
  return launch_ex(select_kernel, grid, dim3(kSelThreads), size_t(smem), static_cast<cudaStream_t>(stream),
                   pdl, 1, a) == cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

extern "C" sa_status sa_select_topk(const float* scores, int32_t max_pages, const sa_batch* batch,
                                    int32_t page_size, int32_t num_kv_heads, int32_t topk,
                                    int32_t* sel_idx, int32_t* sel_cnt, int32_t* dev_status,
                                    void* stream) {
  return sa::select_impl(scores, max_pages, batch, page_size, num_kv_heads, topk, 0, 1, sel_idx,
                         sel_cnt, dev_status, stream, false);
}

extern "C" sa_status sa_select_topk_reserved(const float* scores, int32_t max_pages,
                                             const sa_batch* batch, int32_t page_size,
                                             int32_t num_kv_heads, int32_t topk, int32_t n_bos,
                                             int32_t n_eos, int32_t* sel_idx, int32_t* sel_cnt,
                                             int32_t* dev_status, void* stream) {
  return sa::select_impl(scores, max_pages, batch, page_size, num_kv_heads, topk, n_bos, n_eos,
                         sel_idx, sel_cnt, dev_status, stream, false);
}
