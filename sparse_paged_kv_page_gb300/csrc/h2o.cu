// sa_h2o_update: token-level H2O -- fold this step's attention probabilities
// into the bf16 heavy-hitter scores, then evict above budget.
//
// "flow: add H2O sparse attention" (vortex_torch PR 6), "Token-level
// variants" points 1 and 3: accumulate softmax probabilities (not logits) in a
// bf16 accumulator with multiplicative decay, out = attn + decay * old.
// "H2O -- Cumulative Attention-Mass Heavy-Hitter Oracle Eviction"
// (VeloxQuant-MLX), "Parameters" and "How it works": the first n_sink and the
// newest `grace` retained tokens are protected; above budget the lowest score
// among the rest is evicted (argmin, first index on ties, i.e. the lowest
// position since the list is ascending); the cache ends at most at budget.
//
// One CTA per (KV head, request). Fold: p_bar_j = mean_g exp(z_gj - lse_g) in
// float32; hh = decay * hh + p_bar as one float64 fma rounded once to bf16.
// sa_h2o_update_window follows the reserved windows of the vortex follow-up
// comment ("Two things I had to fix"): the protected entries (the first n_sink
// and the last grace) receive nothing and the softmax is normalised over the
// entries between them, lse_g replaced by their own log-sum-exp.
// Evict: scores are fixed within the step, so evicting the minimum one at a
// time until |R| = budget removes exactly the m = |R| - budget smallest
// (score, position) pairs of the eligible window [n_sink, |R| - grace) (the
// window's ends do not move as entries before them leave). A 2-pass radix
// select over 16-bit score keys finds the m-th smallest key K and how many
// entries equal to K leave (the lowest-positioned ones); block prefix sums
// compact the survivors in order.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

constexpr int kH2oThreads = 512;
constexpr int kH2oMaxCap = 32768;

struct H2oArgs {
  const int32_t* bt;
  const float* logits;
  const float* lse;
  uint16_t* hh;
  int32_t* ret_pos;
  int32_t* ret_cnt;
  int32_t* evicted;
  int32_t* evicted_cnt;
  int32_t* status;
  int H, H_q, G, bt_stride, logits_stride, num_slots, cap, budget, n_sink, grace;
  float decay;
  int window;      // softmax over the unprotected entries only, the protected ones get 0
};

__global__ void __launch_bounds__(kH2oThreads) h2o_kernel(H2oArgs a) {
  extern __shared__ uint8_t sm[];
  int32_t* s_pos = reinterpret_cast<int32_t*>(sm);
  uint16_t* s_key = reinterpret_cast<uint16_t*>(s_pos + a.cap);
  __shared__ int hist[256];
  __shared__ int scan_tmp[32];
  __shared__ int s_digit, s_below;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int unit = b * a.H + h;
  int n = a.ret_cnt[unit];
  if (n < 0 || n > a.cap) {
    if (tid == 0) flag(a.status, SA_DEV_BAD_COUNT);
    n = n < 0 ? 0 : a.cap;
  }
  int32_t* rp = a.ret_pos + int64_t(unit) * a.cap;
  const float inv_g = 1.0f / float(a.G);
  const double decay = double(a.decay);

  // Windowed mode: each query head's log-sum-exp over the unprotected
  // entries [n_sink, n - grace) only; warp g (< G <= 16) reduces head g.
  __shared__ float s_lse_w[16];
  const int wlo = a.n_sink, whi = n - a.grace;
  if (a.window) {
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < a.G) {
      const float* zr = a.logits + (int64_t(b) * a.H_q + h * a.G + warp) * a.logits_stride;
      float m = -INFINITY;
      for (int j = wlo + lane; j < whi; j += 32) m = fmaxf(m, zr[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      float sum = 0.f;
      if (m > -INFINITY)
        for (int j = wlo + lane; j < whi; j += 32) sum += expf(zr[j] - m);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
      if (lane == 0) s_lse_w[warp] = sum > 0.f ? m + logf(sum) : INFINITY;   // +inf: p = 0
    }
    __syncthreads();
  }

  // fold
  for (int j = tid; j < n; j += kH2oThreads) {
    const int pos = rp[j];
    s_pos[j] = pos;
    float pb = 0.f;
    if (!a.window || (j >= wlo && j < whi)) {
      for (int g = 0; g < a.G; ++g) {
        const int hq = h * a.G + g;
        const float z = a.logits[(int64_t(b) * a.H_q + hq) * a.logits_stride + j];
        pb += expf(z - (a.window ? s_lse_w[g] : a.lse[int64_t(b) * a.H_q + hq]));
      }
    }
    pb *= inv_g;
    uint16_t nw = 0xffffu;
    if (pos < 0 || pos >= a.bt_stride) {
      flag(a.status, SA_DEV_BAD_BLOCK);
    } else {
      const int slot = a.bt[int64_t(b) * a.bt_stride + pos];
      if (slot < 0 || slot >= a.num_slots) {
        flag(a.status, SA_DEV_BAD_BLOCK);
      } else {
        uint16_t* hp = a.hh + int64_t(slot) * a.H + h;
        const double old = double(Elem<__nv_bfloat16>::to_f(*hp));
        nw = round_f64<8, -126, 127>(fma(decay, old, double(pb)));
        *hp = nw;
      }
    }
    s_key[j] = uint16_t(bf16_key(nw));
  }
  __syncthreads();

  const int m = n - a.budget;
  if (m <= 0) {
    if (tid == 0 && a.evicted_cnt) a.evicted_cnt[unit] = 0;
    return;
  }
  const int lo = a.n_sink, hi = n - a.grace;     // eligible list indices [lo, hi)

  // radix select of the m-th smallest key in [lo, hi)
  uint32_t prefix = 0, mask = 0;
  int remaining = m;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = 8 - 8 * pass;
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int j0 = lo; j0 < hi; j0 += kH2oThreads) {           // warp-uniform trip count
      const int j = j0 + tid;
      int bin = -1;
      if (j < hi) {
        const uint32_t k = s_key[j];
        if ((k & mask) == prefix) bin = int((k >> shift) & 255u);
      }
      warp_hist_add(hist, bin);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 8l .. 8l+7, scanned upwards
      int c[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { c[q] = hist[8 * tid + q]; sum += c[q]; }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (tid >= o) incl += y;
      }
      int run = incl - sum, found = -1, below = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (found < 0 && run < remaining && remaining <= run + c[q]) { found = 8 * tid + q; below = run; }
        run += c[q];
      }
      const unsigned bm = __ballot_sync(kFull, found >= 0);
      const int src = bm ? __ffs(bm) - 1 : 0;
      const int d = __shfl_sync(kFull, found, src), bl = __shfl_sync(kFull, below, src);
      if (tid == 0) { s_digit = d; s_below = bl; }
    }
    __syncthreads();
    const int d = s_digit;
    remaining -= s_below;
    prefix |= uint32_t(d) << shift;
    mask |= 255u << shift;
    const bool whole = hist[d] == remaining;
    __syncthreads();
    if (whole) break;
  }

  // evict: eligible and ((key & mask) < prefix or (== prefix among the first `remaining`))
  const int per = (n + kH2oThreads - 1) / kH2oThreads;
  const int c0 = min(n, tid * per), c1 = min(n, c0 + per);
  int eq_local = 0;
  for (int j = c0; j < c1; ++j)
    eq_local += (j >= lo && j < hi && (uint32_t(s_key[j]) & mask) == prefix);
  int total;
  const int eq_before = block_exclusive_scan<kH2oThreads>(eq_local, scan_tmp, &total);
  int keep_local = 0;
  {
    int e = eq_before;
    for (int j = c0; j < c1; ++j) {
      bool ev = false;
      if (j >= lo && j < hi) {
        const uint32_t k = uint32_t(s_key[j]) & mask;
        if (k < prefix) ev = true;
        else if (k == prefix) { ev = e < remaining; ++e; }
      }
      keep_local += !ev;
    }
  }
  const int keep_before = block_exclusive_scan<kH2oThreads>(keep_local, scan_tmp, &total);
  {
    int e = eq_before, o = keep_before, x = c0 - keep_before;   // x: evicted before c0
    for (int j = c0; j < c1; ++j) {
      bool ev = false;
      if (j >= lo && j < hi) {
        const uint32_t k = uint32_t(s_key[j]) & mask;
        if (k < prefix) ev = true;
        else if (k == prefix) { ev = e < remaining; ++e; }
      }
      if (ev) {
        if (a.evicted) a.evicted[int64_t(unit) * a.cap + x] = s_pos[j];
        ++x;
      } else {
        rp[o++] = s_pos[j];
      }
    }
  }
  if (tid == 0) {
    a.ret_cnt[unit] = n - m;
    if (a.evicted_cnt) a.evicted_cnt[unit] = m;
  }
}

int g_h2o_smem[64];

}  // namespace
}  // namespace sa

static sa_status h2o_update(const sa_batch* batch, int32_t num_kv_heads, int32_t num_q_heads,
                                   const float* logits, int32_t logits_stride, const float* lse,
                                   void* hh, int32_t num_slots, int32_t* ret_pos, int32_t* ret_cnt,
                                   int32_t ret_cap, int32_t budget, int32_t n_sink, int32_t grace,
                                   float decay, int32_t* evicted, int32_t* evicted_cnt,
                                   int32_t* dev_status, void* stream, int window) {
  using namespace sa;
  sa_status st = check_batch(batch);
  if (st != SA_OK) return st;
  if (!logits || !lse || !hh || !ret_pos || !ret_cnt) return SA_ERR_INVALID_ARG;
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads) return SA_ERR_INVALID_ARG;
  if (ret_cap <= 0 || logits_stride < ret_cap || num_slots <= 0) return SA_ERR_INVALID_ARG;
  if (n_sink < 0 || grace < 0 || budget <= n_sink + grace) return SA_ERR_INVALID_ARG;
  if (!(decay > 0.f && decay <= 1.f)) return SA_ERR_INVALID_ARG;
  if (ret_cap > kH2oMaxCap) return SA_ERR_UNSUPPORTED;
  if (window && num_q_heads / num_kv_heads > 16) return SA_ERR_UNSUPPORTED;
  H2oArgs a;
  a.bt = batch->block_table; a.logits = logits; a.lse = lse; a.hh = static_cast<uint16_t*>(hh);
  a.ret_pos = ret_pos; a.ret_cnt = ret_cnt; a.evicted = evicted; a.evicted_cnt = evicted_cnt;
  a.status = dev_status; a.H = num_kv_heads; a.H_q = num_q_heads; a.G = num_q_heads / num_kv_heads;
  a.bt_stride = batch->bt_stride; a.logits_stride = logits_stride; a.num_slots = num_slots;
  a.cap = ret_cap; a.budget = budget; a.n_sink = n_sink; a.grace = grace; a.decay = decay;
  a.window = window;
  const int smem = ret_cap * 6 + 16;
  if (!ensure_smem(h2o_kernel, smem, g_h2o_smem)) return SA_ERR_CUDA;
  dim3 grid(unsigned(num_kv_heads), unsigned(batch->batch));
  h2o_kernel<<<grid, kH2oThreads, smem, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

extern "C" sa_status sa_h2o_update(const sa_batch* batch, int32_t num_kv_heads, int32_t num_q_heads,
                                   const float* logits, int32_t logits_stride, const float* lse,
                                   void* hh, int32_t num_slots, int32_t* ret_pos, int32_t* ret_cnt,
                                   int32_t ret_cap, int32_t budget, int32_t n_sink, int32_t grace,
                                   float decay, int32_t* evicted, int32_t* evicted_cnt,
                                   int32_t* dev_status, void* stream) {
  return h2o_update(batch, num_kv_heads, num_q_heads, logits, logits_stride, lse, hh, num_slots,
                    ret_pos, ret_cnt, ret_cap, budget, n_sink, grace, decay, evicted, evicted_cnt,
                    dev_status, stream, 0);
}

extern "C" sa_status sa_h2o_update_window(const sa_batch* batch, int32_t num_kv_heads,
                                          int32_t num_q_heads, const float* logits,
                                          int32_t logits_stride, const float* lse, void* hh,
                                          int32_t num_slots, int32_t* ret_pos, int32_t* ret_cnt,
                                          int32_t ret_cap, int32_t budget, int32_t n_sink,
                                          int32_t grace, float decay, int32_t* evicted,
                                          int32_t* evicted_cnt, int32_t* dev_status, void* stream) {
  return h2o_update(batch, num_kv_heads, num_q_heads, logits, logits_stride, lse, hh, num_slots,
                    ret_pos, ret_cnt, ret_cap, budget, n_sink, grace, decay, evicted, evicted_cnt,
                    dev_status, stream, 1);
}
