// sa_select_topk: the pages each (request, KV head) attends.
//
// "EntmaxKV" README, "How it works", "Top-k": keep topk pages, the budget
// counting pages and including the always-attended tail page. With n pages:
// n <= topk keeps all; otherwise the tail n-1 plus the topk-1 best of pages
// 0..n-2 by (score descending, index ascending); -0 == +0; NaN ranks last.
//
// One 1024-thread CTA per (KV head, request). Scores become order-preserving
// 32-bit keys in shared memory; a most-significant-digit radix select
// (12-, 12- and 8-bit digits, early exit once a digit bin is taken whole) finds the
// key K of the (topk-1)-th best candidate and how many candidates equal to K
// to keep; those are the lowest-indexed ones. Two block-wide prefix sums in
// page order then give each kept page its slot, so the output is ascending
// without sorting and the result is deterministic.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

#ifndef SA_SELECT_THREADS
#define SA_SELECT_THREADS 1024
#endif
constexpr int kSelThreads = SA_SELECT_THREADS;
constexpr int kBpt = 4096 / kSelThreads;   // histogram bins owned per thread in the digit search
static_assert(4096 % kSelThreads == 0, "threads must divide the 4096 bins");
constexpr int kSelMaxPages = 45056;      // keys in shared memory next to a 16 KB histogram

struct SelArgs {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* sel_idx;
  int32_t* sel_cnt;
  int32_t* status;
  int H, ps, max_pages, topk;
};

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[4096];
  __shared__ int scan_tmp[32];
  __shared__ int s_digit, s_above;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int unit = b * a.H + h;
  pdl_wait();                                  // scores and lengths of this step are final
  pdl_trigger();                               // the decode may start its prologue
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
  const int kprime = a.topk - 1;                 // best candidates besides the tail
  const int nc = n - 1;                          // candidates 0 .. n-2
  if (kprime == 0) {
    if (tid == 0) { out[0] = n - 1; a.sel_cnt[unit] = 1; }
    return;
  }
  const float* sc = a.scores + int64_t(unit) * a.max_pages;
  for (int i0 = 0; i0 < nc; i0 += 8 * kSelThreads) {      // 8 independent loads per thread
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelThreads + tid;
      v[u] = i < nc ? sc[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelThreads + tid;
      if (i < nc) keys[i] = f32_key(v[u]);
    }
  }

  // Radix select from the most significant digit: 12, 12 and 8 bits. (The top
  // byte of a float key is the sign and high exponent bits -- a 12-bit first
  // digit also takes three mantissa bits, so the first pass already splits
  // typical score distributions into many bins.)
  uint32_t prefix = 0, mask = 0;
  int remaining = kprime;                        // still to take among keys matching prefix
  for (int pass = 0; pass < 3; ++pass) {
    const int width = pass < 2 ? 12 : 8;
    const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
    const int nbins = 1 << width;
    for (int i = tid; i < nbins; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < nc; i += kSelThreads) {
      const uint32_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & uint32_t(nbins - 1)], 1);
    }
    __syncthreads();
    // thread t owns bins nbins-1-kBpt*t-j (j < kBpt), i.e. scanned from the top
    int c[kBpt], sum = 0;
#pragma unroll
    for (int j = 0; j < kBpt; ++j) {
      const int bin = nbins - 1 - kBpt * tid - j;
      c[j] = bin >= 0 ? hist[bin] : 0;
      sum += c[j];
    }
    int total;
    int run = block_exclusive_scan<kSelThreads>(sum, scan_tmp, &total);
#pragma unroll
    for (int j = 0; j < kBpt; ++j) {
      if (run < remaining && remaining <= run + c[j]) { s_digit = nbins - 1 - kBpt * tid - j; s_above = run; }
      run += c[j];
    }
    __syncthreads();
    const int d = s_digit;
    remaining -= s_above;
    prefix |= uint32_t(d) << shift;
    mask |= uint32_t(nbins - 1) << shift;
    const bool whole = hist[d] == remaining;
    __syncthreads();                             // everyone has read hist before it is reset
    if (whole) break;
  }

  // keep: (key & mask) > prefix, or == prefix among the first `remaining` in page order
  const int per = (nc + kSelThreads - 1) / kSelThreads;
  const int c0 = min(nc, tid * per), c1 = min(nc, c0 + per);
  int eq_local = 0;
  for (int i = c0; i < c1; ++i) eq_local += (keys[i] & mask) == prefix;
  int total;
  const int eq_before = block_exclusive_scan<kSelThreads>(eq_local, scan_tmp, &total);
  int take_local = 0;
  {
    int e = eq_before;
    for (int i = c0; i < c1; ++i) {
      const uint32_t k = keys[i] & mask;
      if (k > prefix) ++take_local;
      else if (k == prefix) { take_local += e < remaining; ++e; }
    }
  }
  const int take_before = block_exclusive_scan<kSelThreads>(take_local, scan_tmp, &total);
  {
    int e = eq_before, o = take_before;
    for (int i = c0; i < c1; ++i) {
      const uint32_t k = keys[i] & mask;
      bool take = false;
      if (k > prefix) take = true;
      else if (k == prefix) { take = e < remaining; ++e; }
      if (take && o < kprime) out[o++] = i;
    }
  }
  if (tid == 0) {
    out[kprime] = n - 1;                         // the tail is the largest index
    a.sel_cnt[unit] = a.topk;
  }
}

int g_sel_smem[64];

}  // namespace
}  // namespace sa

sa_status sa::select_impl(const float* scores, int32_t max_pages, const sa_batch* batch,
                         int32_t page_size, int32_t num_kv_heads, int32_t topk, int32_t* sel_idx,
                         int32_t* sel_cnt, int32_t* dev_status, void* stream, bool pdl) {
  using namespace sa;
  sa_status st = check_batch(batch);
  if (st != SA_OK) return st;
  if (!scores || !sel_idx || !sel_cnt || max_pages <= 0 || num_kv_heads <= 0 || topk <= 0)
    return SA_ERR_INVALID_ARG;
  if (!is_pow2(page_size) || page_size > 128) return SA_ERR_UNSUPPORTED;
  if (max_pages > kSelMaxPages) return SA_ERR_UNSUPPORTED;
  SelArgs a;
  a.scores = scores; a.seq_lens = batch->seq_lens; a.sel_idx = sel_idx; a.sel_cnt = sel_cnt;
  a.status = dev_status; a.H = num_kv_heads; a.ps = page_size; a.max_pages = max_pages;
  a.topk = topk;
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
  return sa::select_impl(scores, max_pages, batch, page_size, num_kv_heads, topk, sel_idx, sel_cnt,
                         dev_status, stream, false);
}
