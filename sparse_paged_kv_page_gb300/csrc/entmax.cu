// sa_sparse_decode_entmax: attention over the selected pages with alpha-entmax
// in place of the softmax.
//
// "EntmaxKV" README, "How it works" and "Quick start": the selected pages are
// attended exactly, the normaliser being alpha-entmax (alpha = 1.5 by
// default; 1.5 and 2 have closed forms): with a_j = (alpha - 1) z_j, z_j the
// scaled logits of the selection, p_j = (a_j - tau)_+ ^ (1 / (alpha - 1)) and
// tau fixed by sum_j p_j = 1.
//
// Four launches:
//  (1) the decode kernel in its logits-only mode writes z for every selected
//      token (K is read; V is not);
//  (2) entmax_tau_kernel, one CTA per (request, query head), finds tau.
//      f(tau) = sum_j (a_j - tau)_+^r - 1 (r = 1 / (alpha - 1) >= 1) is convex
//      and decreasing, and f(a_max - 1) >= 0 (the top entry alone gives 1), so
//      Newton's method from a_max - 1 rises monotonically to the root. For
//      alpha = 2 and 1.5 each iterate's support {a_j > tau} also gives the
//      closed-form root of that support; once that root lies below every
//      member of the support it is the exact tau (the rule "largest support
//      whose threshold stays below its smallest member"). Sums are float64,
//      centred on the current iterate. Since tau >= a_max - 1, only entries
//      above a_max - 1 can enter the support: those are gathered first (in
//      row order) and one warp iterates over them alone;
//  (3) entmax_pv_kernel, split over tokens, one CTA per (split, request, KV
//      head): each warp tests 32 tokens at a time against the G heads' tau
//      and loads V rows only for tokens some head of the group keeps
//      (entmax is sparse), accumulating sum_j p_j v_j and sum_j p_j in fp32;
//  (4) entmax_finish_kernel adds the splits in a fixed order and divides by
//      sum_j p_j (1 up to the rounding of tau), writing bf16/fp16.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

constexpr int kTauThreads = 256;
constexpr int kTauWarps = kTauThreads / 32;
constexpr int kPvThreads = 256;
constexpr int kPvWarps = kPvThreads / 32;
constexpr int kTauMaxIter = 100;
constexpr int kTauCand = 2048;          // candidates one warp solves over

struct EntArgs {
  const void* v;
  const int32_t* bt;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* cnt;
  const float* logits;   // [B, H_q, logits_stride]
  float* tau;            // [B, H_q] (NaN: no token with a finite logit)
  float* tau_out;        // optional copy for the caller
  float* part_o;         // [B, H_q, nsplit, D]
  float* part_l;         // [B, H_q, nsplit]
  void* out;
  int32_t* status;
  int H_kv, H_q, G, ps, ps_shift, num_blocks, bt_stride, sel_stride, logits_stride, nsplit, ent_cap;
  float alpha;
};

// 0: generic alpha (Newton only), 1: alpha = 1.5, 2: alpha = 2
__host__ __device__ inline int alpha_kind(float alpha) {
  return alpha == 2.0f ? 2 : (alpha == 1.5f ? 1 : 0);
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ double warp_min_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmin(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Newton's method with the closed-form finish over the values x[0, m),
// entries <= skip never in the support, from tau (back to tau_left = a_max - 1,
// always left of the root, if tau turns out to lie right of it). kBlock: all threads of the CTA share
// the work (float64 sums through shared memory); else one warp alone. Every
// participating thread returns the same tau.
template <bool kBlock>
__device__ double solve_tau(const float* x, int m, double tau, double tau_left, float skip,
                            int kind, double r, double (*red)[kTauWarps][4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = kBlock ? int(threadIdx.x) : lane;
  const int stride = kBlock ? kTauThreads : 32;
  bool restarted = tau == tau_left;
  for (int it = 0; it < kTauMaxIter; ++it) {
    // over the support {a > tau}: count, sum d^r, sum d^(r-1), min d  (d = a - tau)
    double k = 0.0, p0 = 0.0, p1 = 0.0, mn = INFINITY;
    for (int j = t0; j < m; j += stride) {
      const float xf = x[j];
      if (!(xf > skip)) continue;
      const double d = double(xf) - tau;
      if (d > 0.0) {
        k += 1.0;
        if (kind == 2) { p0 += d; p1 += 1.0; }
        else if (kind == 1) { p0 += d * d; p1 += d; }
        else { const double t = pow(d, r - 1.0); p0 += t * d; p1 += t; }
        mn = fmin(mn, d);
      }
    }
    k = warp_sum_d(k); p0 = warp_sum_d(p0); p1 = warp_sum_d(p1); mn = warp_min_d(mn);
    if constexpr (kBlock) {
      double(*rb)[4] = red[it & 1];                       // alternate buffers: one barrier a round
      if (lane == 0) { rb[warp][0] = k; rb[warp][1] = p0; rb[warp][2] = p1; rb[warp][3] = mn; }
      __syncthreads();
      k = rb[0][0]; p0 = rb[0][1]; p1 = rb[0][2]; mn = rb[0][3];
#pragma unroll
      for (int w = 1; w < kTauWarps; ++w) {
        k += rb[w][0]; p0 += rb[w][1]; p1 += rb[w][2]; mn = fmin(mn, rb[w][3]);
      }
    }
    if (k <= 0.0) break;                                  // (cannot happen below the root)
    if (kind != 0) {
      // the closed-form root of this support, as an offset from tau
      double delta;
      if (kind == 2) {
        delta = (p0 - 1.0) / k;                           // sum d = 1 + k delta
      } else {
        const double disc = fmax(p1 * p1 - k * (p0 - 1.0), 0.0);   // k delta^2 - 2 delta sum d + sum d^2 - 1 = 0
        delta = (p1 - sqrt(disc)) / k;
      }
      if (delta >= 0.0 && delta < mn) { tau += delta; break; }   // every member stays positive: exact
    }
    const double f = p0 - 1.0;
    if (f < -1e-12 && !restarted) {                       // started right of the root: go left
      tau = tau_left;
      restarted = true;
      continue;
    }
    if (f <= 0.0) break;                                  // at the root up to rounding
    const double step = f / (r * p1);
    if (kind == 0 && step <= 1e-15 * fmax(1.0, fabs(tau))) break;
    tau += step;
  }
  return tau;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ float warp_min_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ double warp_max_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// One warp, float32: Newton from a_max - 1 (with the closed-form shortcut for
// alpha 1.5 / 2) to locate the support. Only a first estimate: the float64
// check below decides.
__device__ float tau_estimate(const float* x, int m, float tau, int kind, float r) {
  const int lane = threadIdx.x & 31;
  for (int it = 0; it < kTauMaxIter; ++it) {
    float k = 0.f, p0 = 0.f, p1 = 0.f, mn = INFINITY;
    for (int j = lane; j < m; j += 32) {
      const float d = x[j] - tau;
      if (d > 0.f) {
        k += 1.f;
        if (kind == 2) { p0 += d; p1 += 1.f; }
        else if (kind == 1) { p0 += d * d; p1 += d; }
        else { const float t = powf(d, r - 1.f); p0 += t * d; p1 += t; }
        mn = fminf(mn, d);
      }
    }
    k = warp_sum_f(k); p0 = warp_sum_f(p0); p1 = warp_sum_f(p1); mn = warp_min_f(mn);
    if (k <= 0.f) break;
    if (kind != 0) {
      float delta;
      if (kind == 2) delta = (p0 - 1.f) / k;
      else delta = (p1 - sqrtf(fmaxf(p1 * p1 - k * (p0 - 1.f), 0.f))) / k;
      if (delta >= 0.f && delta < mn) return tau + delta;
    }
    const float f = p0 - 1.f;
    if (f <= 0.f) break;
    const float step = f / (r * p1);
    if (step <= 1e-7f * fmaxf(1.f, fabsf(tau))) break;
    tau += step;
  }
  return tau;
}

// One warp, float64, alpha 1.5 / 2: the closed-form root tau_c of the support
// S = {a > t}. It is the exact threshold when S is consistent with it: every
// member above tau_c and every other entry at or below it (then S = {a > tau_c}
// and sum_S (a - tau_c)^r = 1, whose root is unique).
__device__ bool tau_exact_check(const float* x, int m, double t, int kind, double* tau) {
  const int lane = threadIdx.x & 31;
  double k = 0.0, s1 = 0.0, s2 = 0.0, mn = INFINITY, mo = -INFINITY;
  for (int j = lane; j < m; j += 32) {
    const double d = double(x[j]) - t;
    if (d > 0.0) { k += 1.0; s1 += d; s2 += d * d; mn = fmin(mn, d); }
    else mo = fmax(mo, d);
  }
  k = warp_sum_d(k); s1 = warp_sum_d(s1); s2 = warp_sum_d(s2);
  mn = warp_min_d(mn); mo = warp_max_d(mo);
  if (k <= 0.0) return false;
  const double delta = kind == 2 ? (s1 - 1.0) / k
                                 : (s1 - sqrt(fmax(s1 * s1 - k * (s2 - 1.0), 0.0))) / k;
  if (!(delta < mn && delta >= mo)) return false;
  *tau = t + delta;
  return true;
}

__global__ void __launch_bounds__(kTauThreads) entmax_tau_kernel(EntArgs a) {
  extern __shared__ float s_a[];                          // (alpha - 1) z of the row
  __shared__ float s_c[kTauCand];                         // the candidates, in row order
  __shared__ double red[2][kTauWarps][4];
  __shared__ float redf[kTauWarps];
  __shared__ int redi[kTauWarps];
  const int gq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int c = a.cnt[b * a.H_kv + gq / a.G];
  c = max(0, min(c, a.sel_stride));
  const int n = c << a.ps_shift;
  const float* z = a.logits + (int64_t(b) * a.H_q + gq) * a.logits_stride;
  const float am1 = a.alpha - 1.0f;
  float mx = -INFINITY;
  for (int j = tid; j < n; j += kTauThreads) {
    const float v = z[j];
    const float x = (v > -INFINITY && v < INFINITY) ? am1 * v : -INFINITY;  // NaN / inf never enter
    s_a[j] = x;
    mx = fmaxf(mx, x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  if (lane == 0) redf[warp] = mx;
  __syncthreads();
  mx = redf[0];
#pragma unroll
  for (int w = 1; w < kTauWarps; ++w) mx = fmaxf(mx, redf[w]);
  const int64_t row = int64_t(b) * a.H_q + gq;
  if (!(mx > -INFINITY)) {
    if (tid == 0) {
      a.tau[row] = __int_as_float(0x7fc00000);
      if (a.tau_out) a.tau_out[row] = __int_as_float(0x7fc00000);
    }
    return;
  }
  const int kind = alpha_kind(a.alpha);
  const double r = 1.0 / double(am1);
  // tau never drops below a_max - 1, so only a > a_max - 1 can be in the
  // support: gather those (with a margin for the float rounding) in row order
  const float lo = (mx - 1.0f) - 1e-6f * (1.0f + fabsf(mx));
  const int per = (n + kTauThreads - 1) / kTauThreads;
  const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
  int mine = 0;
  for (int j = j0; j < j1; ++j) mine += s_a[j] > lo;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) redi[warp] = incl;
  __syncthreads();
  int off = incl - mine, m = 0;
#pragma unroll
  for (int w = 0; w < kTauWarps; ++w) {
    if (w < warp) off += redi[w];
    m += redi[w];
  }
  double tau;
  if (m <= kTauCand) {
    for (int j = j0; j < j1; ++j)
      if (s_a[j] > lo) s_c[off++] = s_a[j];
    __syncthreads();
    if (warp != 0) return;
    const float est = tau_estimate(s_c, m, mx - 1.0f, kind, float(r));
    if (kind == 0 || !tau_exact_check(s_c, m, double(est), kind, &tau)) {
      // generic alpha, or a support the float32 estimate got wrong: float64
      // Newton from the left (from a_max - 1, or from just below the estimate
      // when that is still left of the root)
      const double t0 = fmax(double(mx) - 1.0, double(est) - 1e-3 * (1.0 + fabs(double(est))));
      tau = solve_tau<false>(s_c, m, t0, double(mx) - 1.0, -INFINITY, kind, r, red);
    }
  } else {
    tau = solve_tau<true>(s_a, n, double(mx) - 1.0, double(mx) - 1.0, lo, kind, r, red);
  }
  if (tid == 0) {
    a.tau[row] = float(tau);
    if (a.tau_out) a.tau_out[row] = float(tau);
  }
}

template <typename T, int D, int kG>
__global__ void __launch_bounds__(kPvThreads, 2) entmax_pv_kernel(EntArgs a) {
  using E = Elem<T>;
  constexpr int DPL = D / 32;                              // dims per lane: 4 (D 128) or 2 (D 64)
  constexpr int kU = kG > 8 ? 4 : 8;                       // V rows in flight per warp
  extern __shared__ float4 smem_f4[];
  float* s_red = reinterpret_cast<float*>(smem_f4);       // [warps][G][D], then [warps][G]
  int2* s_ent = reinterpret_cast<int2*>(s_red + kPvWarps * a.G * (D + 1));
  __shared__ float s_tau[kG];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = a.G;
  if (tid < G) s_tau[tid] = a.tau[int64_t(b) * a.H_q + h * G + tid];
  int c = a.cnt[b * a.H_kv + h];
  c = max(0, min(c, a.sel_stride));
  const int n = c << a.ps_shift;
  const int per = (((n + a.nsplit - 1) / a.nsplit) + 31) & ~31;
  const int t_lo = min(n, split * per), t_hi = min(n, t_lo + per);
  const int L = a.seq_lens[b];
  const int n_pages_req = L > 0 ? (L + a.ps - 1) >> a.ps_shift : 0;
  const int32_t* sel = a.sel + int64_t(b * a.H_kv + h) * a.sel_stride;
  const int32_t* btb = a.bt + int64_t(b) * a.bt_stride;
  // the selection entries this CTA touches, resolved to (block, fill) once
  const int e_lo = t_lo >> a.ps_shift;
  const int e_n = t_hi > t_lo ? min(((t_hi - 1) >> a.ps_shift) - e_lo + 1, a.ent_cap) : 0;
  for (int i = tid; i < e_n; i += kPvThreads) {
    const int page = sel[e_lo + i];
    int blk = -1, fill = 0;
    if (page >= 0 && page < n_pages_req && page < a.bt_stride) {
      const int x = btb[page];
      if (x >= 0 && x < a.num_blocks) { blk = x; fill = min(a.ps, L - (page << a.ps_shift)); }
    }
    s_ent[i] = make_int2(blk, fill);
  }
  __syncthreads();

  const float am1 = a.alpha - 1.0f;
  const int kind = alpha_kind(a.alpha);
  const float r = 1.0f / am1;
  float acc[kG][DPL], psum[kG];
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    psum[g] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[g][d] = 0.f;
  }
  const float* zb = a.logits + (int64_t(b) * a.H_q + int64_t(h) * G) * a.logits_stride;
  const T* vbase = static_cast<const T*>(a.v);
  for (int base = t_lo + warp * 32; base < t_hi; base += kPvWarps * 32) {
    // p of token base + lane for every head of the group
    const int j = base + lane;
    float p[kG];
    bool keep = false;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      p[g] = 0.f;
      if (g < G && j < t_hi) {
        const float zz = zb[int64_t(g) * a.logits_stride + j];
        const float x = am1 * zz - s_tau[g];
        if (zz > -INFINITY && zz < INFINITY && x > 0.f)
          p[g] = kind == 2 ? x : (kind == 1 ? x * x : powf(x, r));
      }
      keep |= p[g] > 0.f;
    }
    // a token whose page / slot does not resolve is dropped (the logits pass flagged it)
    if (keep) {
      const int ei = (j >> a.ps_shift) - e_lo, s = j & (a.ps - 1);
      const int2 en = (ei >= 0 && ei < e_n) ? s_ent[ei] : make_int2(-1, 0);
      if (en.x < 0 || s >= en.y) {
        keep = false;
#pragma unroll
        for (int g = 0; g < kG; ++g) p[g] = 0.f;
      }
    }
#pragma unroll
    for (int g = 0; g < kG; ++g) psum[g] += p[g];
    uint32_t m = __ballot_sync(kFull, keep);
    while (m) {
      int src[kU];
      float vv[kU][DPL];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        src[u] = m ? __ffs(m) - 1 : -1;
        m &= m - 1;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (src[u] >= 0) {
          const int jj = base + src[u];
          const int2 en = s_ent[(jj >> a.ps_shift) - e_lo];
          const int s = jj & (a.ps - 1);
          const T* vrow = vbase + ((int64_t(en.x) * a.H_kv + h) * a.ps + s) * D + lane * DPL;
          if constexpr (DPL == 4) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(vrow));
            vv[u][0] = E::lo(w.x); vv[u][1] = E::hi(w.x); vv[u][2] = E::lo(w.y); vv[u][3] = E::hi(w.y);
          } else {
            const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(vrow));
            vv[u][0] = E::lo(w); vv[u][1] = E::hi(w);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (src[u] >= 0) {
#pragma unroll
          for (int g = 0; g < kG; ++g) {
            const float pg = __shfl_sync(kFull, p[g], src[u]);
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[g][d] = fmaf(pg, vv[u][d], acc[g][d]);
          }
        }
      }
    }
  }
  // the warps' partial sums, added in a fixed order
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    float ps = psum[g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(kFull, ps, o);
    if (g < G) {
#pragma unroll
      for (int d = 0; d < DPL; ++d) s_red[(warp * G + g) * D + lane * DPL + d] = acc[g][d];
      if (lane == 0) s_red[kPvWarps * G * D + warp * G + g] = ps;
    }
  }
  __syncthreads();
  const int64_t prow = (int64_t(b) * a.H_q + int64_t(h) * G) * a.nsplit;   // (b, head h*G, split 0)
  for (int idx = tid; idx < G * D; idx += kPvThreads) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kPvWarps; ++w) sum += s_red[w * G * D + idx];
    const int g = idx / D, d = idx % D;
    a.part_o[((prow + int64_t(g) * a.nsplit) + split) * D + d] = sum;
  }
  if (tid < G) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kPvWarps; ++w) sum += s_red[kPvWarps * G * D + w * G + tid];
    a.part_l[prow + int64_t(tid) * a.nsplit + split] = sum;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(D) entmax_finish_kernel(EntArgs a) {
  using E = Elem<T>;
  const int gq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int64_t row = int64_t(b) * a.H_q + gq;
  float o = 0.f, l = 0.f;
  for (int s = 0; s < a.nsplit; ++s) {
    o += a.part_o[(row * a.nsplit + s) * D + d];
    l += a.part_l[row * a.nsplit + s];
  }
  const float y = l > 0.f ? o / l : 0.f;                   // no kept token: 0
  reinterpret_cast<uint16_t*>(a.out)[row * D + d] = E::from_f(y);
}

int device_sms() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    sms[dev] = v;
  }
  return sms[dev];
}

struct EntLayout {
  int nsplit, ent_cap;
  size_t logits, tau, part_o, part_l, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// splits: about two CTAs per SM over all (request, KV head) units, at least
// 128 tokens a split
EntLayout ent_layout(int B, int H_kv, int H_q, int D, int ps, int sel_stride, int sms) {
  EntLayout w;
  const int64_t rows = int64_t(sel_stride) * ps;
  const int units = B * H_kv;
  int ns = (2 * sms + units - 1) / units;
  const int64_t by_len = (rows + 127) / 128;
  if (ns > by_len) ns = int(by_len);
  if (ns > 64) ns = 64;
  if (ns < 1) ns = 1;
  w.nsplit = ns;
  const int64_t per = (((rows + ns - 1) / ns) + 31) & ~int64_t(31);
  w.ent_cap = int(per / ps + 2);
  size_t off = 0;
  w.logits = off; off = align256(off + size_t(B) * H_q * rows * sizeof(float));
  w.tau = off;    off = align256(off + size_t(B) * H_q * sizeof(float));
  w.part_o = off; off = align256(off + size_t(B) * H_q * ns * D * sizeof(float));
  w.part_l = off; off = align256(off + size_t(B) * H_q * ns * sizeof(float));
  w.total = off;
  return w;
}

int g_tau_smem[64];
int g_pv_smem[12][64];

template <typename T, int D, int kG>
sa_status launch_pv(const EntArgs& a, dim3 grid, cudaStream_t s, int* attr) {
  const int smem = (kPvWarps * a.G * (D + 1)) * int(sizeof(float)) + a.ent_cap * int(sizeof(int2));
  if (!ensure_smem(entmax_pv_kernel<T, D, kG>, smem, attr)) return SA_ERR_CUDA;
  entmax_pv_kernel<T, D, kG><<<grid, kPvThreads, smem, s>>>(a);
  if (launch_status() != SA_OK) return SA_ERR_CUDA;
  entmax_finish_kernel<T, D><<<dim3(unsigned(a.H_q), grid.z), D, 0, s>>>(a);
  return launch_status();
}

template <typename T, int D>
sa_status launch_pv_g(const EntArgs& a, dim3 grid, cudaStream_t s, int slot) {
  if (a.G <= 4) return launch_pv<T, D, 4>(a, grid, s, g_pv_smem[slot * 3 + 0]);
  if (a.G <= 8) return launch_pv<T, D, 8>(a, grid, s, g_pv_smem[slot * 3 + 1]);
  return launch_pv<T, D, 16>(a, grid, s, g_pv_smem[slot * 3 + 2]);
}

}  // namespace
}  // namespace sa

extern "C" size_t sa_entmax_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t num_q_heads,
                                           int32_t head_dim, int32_t page_size, int32_t sel_stride) {
  using namespace sa;
  if (batch <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      sel_stride <= 0 || num_q_heads % num_kv_heads)
    return 0;
  return ent_layout(batch, num_kv_heads, num_q_heads, head_dim, page_size, sel_stride, device_sms())
      .total;
}

extern "C" sa_status sa_sparse_decode_entmax(const sa_cache* cache, const sa_batch* batch,
                                             const void* q, int32_t num_q_heads,
                                             const int32_t* sel_idx, const int32_t* sel_cnt,
                                             int32_t sel_stride, float alpha, float scale, void* out,
                                             float* tau, float* logits, int32_t logits_stride,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, void* stream) {
  using namespace sa;
  sa_status st = check_cache(cache, true, false);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (!q || !sel_idx || !sel_cnt || !out || sel_stride <= 0) return SA_ERR_INVALID_ARG;
  if (!(alpha > 1.0f && alpha <= 2.0f)) return SA_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return SA_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  if (G > 16) return SA_ERR_UNSUPPORTED;
  const int64_t rows = int64_t(sel_stride) * cache->page_size;
  if (rows * int64_t(sizeof(float)) > 160 * 1024) return SA_ERR_UNSUPPORTED;   // a row of a in shared memory
  if (logits && logits_stride < rows) return SA_ERR_INVALID_ARG;
  const EntLayout w = ent_layout(batch->batch, cache->num_kv_heads, num_q_heads, cache->head_dim,
                                 cache->page_size, sel_stride, device_sms());
  if (!workspace || workspace_bytes < w.total) return SA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* lg = logits ? logits : reinterpret_cast<float*>(ws + w.logits);
  const int lg_stride = logits ? logits_stride : int(rows);
  // (1) the logits of every selected token (K only)
  st = decode_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, sel_stride, scale, out, nullptr, lg,
                   lg_stride, nullptr, 0, dev_status, stream, /*allow_cluster=*/false, /*pdl=*/false,
                   /*per_query_head=*/false, /*logits_only=*/true);
  if (st != SA_OK) return st;
  EntArgs a;
  a.v = cache->v; a.bt = batch->block_table; a.seq_lens = batch->seq_lens; a.sel = sel_idx;
  a.cnt = sel_cnt; a.logits = lg; a.tau = reinterpret_cast<float*>(ws + w.tau); a.tau_out = tau;
  a.part_o = reinterpret_cast<float*>(ws + w.part_o); a.part_l = reinterpret_cast<float*>(ws + w.part_l);
  a.out = out; a.status = dev_status;
  a.H_kv = cache->num_kv_heads; a.H_q = num_q_heads; a.G = G; a.ps = cache->page_size;
  a.ps_shift = log2i(cache->page_size); a.num_blocks = cache->num_blocks;
  a.bt_stride = batch->bt_stride; a.sel_stride = sel_stride; a.logits_stride = lg_stride;
  a.nsplit = w.nsplit; a.ent_cap = w.ent_cap; a.alpha = alpha;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // (2) tau per (request, query head)
  const int tsmem = int(rows * sizeof(float));
  if (!ensure_smem(entmax_tau_kernel, tsmem, g_tau_smem)) return SA_ERR_CUDA;
  entmax_tau_kernel<<<dim3(unsigned(num_q_heads), unsigned(batch->batch)), kTauThreads, tsmem, s>>>(a);
  if ((st = launch_status()) != SA_OK) return st;
  // (3) the kept tokens' sum_j p_j v_j per split, (4) the splits added and normalised
  const dim3 grid(unsigned(w.nsplit), unsigned(cache->num_kv_heads), unsigned(batch->batch));
  const bool bf = cache->dtype == SA_BF16;
  if (cache->head_dim == 128)
    return bf ? launch_pv_g<__nv_bfloat16, 128>(a, grid, s, 0) : launch_pv_g<__half, 128>(a, grid, s, 1);
  return bf ? launch_pv_g<__nv_bfloat16, 64>(a, grid, s, 2) : launch_pv_g<__half, 64>(a, grid, s, 3);
}
