// sa_gauss_select: Gaussian-aware page selection, per query head.
//
// "EntmaxKV" README, "How it works" (Gaussian-aware strategy): each page's
// scores are modelled as a Gaussian from its per-page key statistics (mean
// and std, without touching the cached tokens), the distributional entmax
// constraint is solved for the threshold tau_hat (a single Gaussian for heads
// without ALiBi), and every page whose estimated maximum can cross tau_hat is
// selected; the count adapts to the distribution. The tail page is always
// kept (as the top-k strategy's budget counts it).
//
// Two launches:
//  (1) gauss_moments_kernel: one thread per page of a (request, KV head),
//      reading a whole 32-byte sector of its mean and std rows per step, scale
//      q of the G heads in shared memory; with the page's dimensions taken as
//      independent, a query head's scores z = scale q . k on page p have
//        m_p = sum_d (scale q_d) mean_pd,  v_p = sum_d (scale q_d)^2 std_pd^2.
//  (2) gauss_select_kernel: one CTA per (request, query head). The page
//      mixture's moments N = sum f_p, M = sum f m / N, V = sum f (v + m^2) / N
//      - M^2 (compensated float32 per thread, float64 across threads) define
//      N(M, V); tau_hat solves N E[((alpha - 1) Z - tau)_+^(1/(alpha - 1))] = 1
//      with the truncated-normal closed forms (alpha 1.5 / 2), by Newton's
//      method from (alpha - 1) M - 1, which Jensen's inequality puts left of
//      the root of this convex, decreasing function. Page p is kept when
//      (alpha - 1)(m_p + sqrt(2 ln f_p) sqrt(v_p)) > tau_hat (sqrt(2 ln f)
//      bounds the expected maximum of f Gaussian scores) or it is the tail;
//      the kept pages are written in page order (per-warp segments, one
//      exchange of counts).
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

constexpr int kMomThreads = 128;
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

struct GaussArgs {
  const void* meta;
  const void* kstd;
  const void* q;
  const int32_t* bt;
  const int32_t* seq_lens;
  float2* mom;           // [B, H_q, max_pages]: (m, v); m = -inf for a page that does not resolve
  int32_t* sel;          // [B, H_q, sel_stride]
  int32_t* cnt;          // [B, H_q]
  float* tau_hat;        // nullable [B, H_q]
  int32_t* status;
  int H_kv, H_q, G, ps, ps_shift, num_blocks, bt_stride, max_pages, sel_stride;
  int est_in_smem;       // the selection kernel keeps every page's estimate in shared memory
  float scale, alpha;
};

template <typename T, int D, int kG>
__global__ void __launch_bounds__(kMomThreads) gauss_moments_kernel(GaussArgs a) {
  using E = Elem<T>;
  __shared__ float4 s_q[kG][D / 4];      // scale * q
  const int h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int G = a.G;
  const uint16_t* qb = static_cast<const uint16_t*>(a.q) + (int64_t(b) * a.H_q + int64_t(h) * G) * D;
  for (int i = tid; i < G * D; i += kMomThreads) {
    reinterpret_cast<float*>(s_q)[i] = a.scale * E::lo(uint32_t(qb[i]));
  }
  __syncthreads();
  const int L = a.seq_lens[b];
  const int n = min(L > 0 ? (L + a.ps - 1) >> a.ps_shift : 0, a.max_pages);
  const int p = blockIdx.x * kMomThreads + tid;
  if (p >= n) return;
  float m[kG], v[kG];
#pragma unroll
  for (int g = 0; g < kG; ++g) m[g] = v[g] = 0.f;
  const int blk = a.bt[int64_t(b) * a.bt_stride + p];
  const int64_t mrow = int64_t(b) * a.H_q + int64_t(h) * G;
  if (blk < 0 || blk >= a.num_blocks) {
    flag(a.status, SA_DEV_BAD_BLOCK);
    for (int g = 0; g < G; ++g) a.mom[(mrow + g) * a.max_pages + p] = make_float2(-INFINITY, 0.f);
    return;
  }
  const uint4* mu = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.meta) +
                                                   ((int64_t(blk) * a.H_kv + h) * 3 + 2) * D);
  const uint4* sd = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.kstd) +
                                                   (int64_t(blk) * a.H_kv + h) * D);
  // a full 32-byte sector of each row per step (16 dimensions)
#pragma unroll 2
  for (int c = 0; c < D / 16; ++c) {
    const uint4 um0 = __ldg(mu + 2 * c), um1 = __ldg(mu + 2 * c + 1);
    const uint4 us0 = __ldg(sd + 2 * c), us1 = __ldg(sd + 2 * c + 1);
    const uint32_t wm[8] = {um0.x, um0.y, um0.z, um0.w, um1.x, um1.y, um1.z, um1.w};
    const uint32_t ws[8] = {us0.x, us0.y, us0.z, us0.w, us1.x, us1.y, us1.z, us1.w};
    float xm[16], xs[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      xm[2 * i] = E::lo(wm[i]); xm[2 * i + 1] = E::hi(wm[i]);
      const float s0 = E::lo(ws[i]), s1 = E::hi(ws[i]);
      xs[2 * i] = s0 * s0; xs[2 * i + 1] = s1 * s1;
    }
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      if (g < G) {
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4) {
          const float4 qv = s_q[g][4 * c + h4];
          const float qq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            m[g] = fmaf(qq[i], xm[4 * h4 + i], m[g]);
            v[g] = fmaf(qq[i] * qq[i], xs[4 * h4 + i], v[g]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < kG; ++g)
    if (g < G) a.mom[(mrow + g) * a.max_pages + p] = make_float2(m[g], v[g]);
}

// s += x with the rounding error carried in c (Kahan-Babuska-Neumaier)
__device__ __forceinline__ void csum(float& s, float& c, float x) {
  const float t = s + x;
  c += fabsf(s) >= fabsf(x) ? (s - t) + x : (x - t) + s;
  s = t;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// E[(A - t)_+^r] and its derivative in t for A ~ N(mu_a, s_a^2), r = 1 / (alpha - 1)
__device__ __forceinline__ void tail_moment(float mu_a, float s_a, float t, bool sparsemax, float& e,
                                            float& de) {
  const float c = mu_a - t;
  if (s_a <= 0.f) {
    const float cp = fmaxf(c, 0.f);
    e = sparsemax ? cp : cp * cp;
    de = sparsemax ? -(c > 0.f ? 1.f : 0.f) : -2.f * cp;
    return;
  }
  const float u = c / s_a;
  const float Phi = 0.5f * erfcf(-u * 0.70710678118654752f);
  const float phi = 0.39894228040143268f * expf(-0.5f * u * u);
  const float m1 = c * Phi + s_a * phi;                    // E[(A - t)_+]
  if (sparsemax) {
    e = m1;
    de = -Phi;
  } else {
    e = (c * c + s_a * s_a) * Phi + c * s_a * phi;         // E[(A - t)_+^2]
    de = -2.f * m1;
  }
}

// the page's estimated maximum score m + sqrt(2 ln f) sqrt(v); kappa_full is
// sqrt(2 ln page_size), every page but the tail being full
__device__ __forceinline__ float est_max(float2 mv, int f, int ps, float kappa_full) {
  const float kappa = f == ps ? kappa_full : (f > 1 ? sqrtf(2.0f * logf(float(f))) : 0.f);
  return mv.x + kappa * sqrtf(fmaxf(mv.y, 0.f));
}

__global__ void __launch_bounds__(kSelThreads) gauss_select_kernel(GaussArgs a) {
  __shared__ double s_red[kSelWarps][3];
  __shared__ int s_cnt[kSelWarps];
  __shared__ float s_tau;
  const int gq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int L = a.seq_lens[b];
  const int n_all = L > 0 ? (L + a.ps - 1) >> a.ps_shift : 0;
  if (n_all > a.max_pages && tid == 0) flag(a.status, SA_DEV_OVERFLOW);
  const int n = min(n_all, a.max_pages);
  const int64_t row = int64_t(b) * a.H_q + gq;
  const float2* mom = a.mom + row * a.max_pages;
  if (n == 0) {
    if (tid == 0) {
      a.cnt[row] = 0;
      if (a.tau_hat) a.tau_hat[row] = __int_as_float(0x7fc00000);
    }
    return;
  }
  // the mixture's moments; each page's estimated maximum kept for the selection
  extern __shared__ float s_est[];                          // [max_pages] when it fits, else unused
  const bool cached = a.est_in_smem;
  const float kappa_full = a.ps > 1 ? sqrtf(2.0f * logf(float(a.ps))) : 0.f;
  float f_s = 0.f, s1 = 0.f, c1 = 0.f, s2 = 0.f, c2 = 0.f;
#pragma unroll 8
  for (int p = tid; p < n; p += kSelThreads) {
    const float2 mv = __ldcg(mom + p);
    const bool ok = mv.x > -INFINITY && mv.x < INFINITY;
    const int fi = min(a.ps, L - (p << a.ps_shift));
    if (cached) s_est[p] = ok ? est_max(mv, fi, a.ps, kappa_full) : -INFINITY;
    if (!ok) continue;
    const float f = float(fi);
    f_s += f;
    csum(s1, c1, f * mv.x);
    csum(s2, c2, f * (mv.y + mv.x * mv.x));
  }
  double dn = warp_sum_d(double(f_s)), d1 = warp_sum_d(double(s1) + double(c1)),
         d2 = warp_sum_d(double(s2) + double(c2));
  if (lane == 0) { s_red[warp][0] = dn; s_red[warp][1] = d1; s_red[warp][2] = d2; }
  __syncthreads();
  if (tid == 0) {
    double N = 0.0, S1 = 0.0, S2 = 0.0;
    for (int w = 0; w < kSelWarps; ++w) { N += s_red[w][0]; S1 += s_red[w][1]; S2 += s_red[w][2]; }
    float tau = -INFINITY;                                  // nothing resolves: only the tail
    if (N > 0.0) {
      const double Md = S1 / N;
      const float M = float(Md), V = float(fmax(S2 / N - Md * Md, 0.0));
      const bool sparsemax = a.alpha == 2.0f;
      const float am1 = a.alpha - 1.0f;
      const float mu_a = am1 * M, s_a = am1 * sqrtf(V), Nf = float(N);
      if (s_a <= 0.f) {
        tau = mu_a - (sparsemax ? 1.0f / Nf : rsqrtf(Nf));  // N (mu_a - tau)^r = 1
      } else {
        tau = mu_a - 1.0f;                                  // left of the root (Jensen)
        for (int it = 0; it < 100; ++it) {
          float e, de;
          tail_moment(mu_a, s_a, tau, sparsemax, e, de);
          const float g = Nf * e - 1.0f;
          if (!(g > 0.f) || !(de < 0.f)) break;
          const float step = -g / (Nf * de);
          tau += step;
          if (step <= 1e-7f * (1.0f + fabsf(tau))) break;
        }
      }
    }
    s_tau = tau;
    if (a.tau_hat) a.tau_hat[row] = tau;
  }
  __syncthreads();
  const float tau = s_tau, am1 = a.alpha - 1.0f;
  auto keep_of = [&](int p) -> bool {
    if (p == n - 1) return true;                            // the tail page
    float e;
    if (cached) {
      e = s_est[p];
    } else {
      const float2 mv = mom[p];
      if (!(mv.x > -INFINITY && mv.x < INFINITY)) return false;
      e = est_max(mv, min(a.ps, L - (p << a.ps_shift)), a.ps, kappa_full);
    }
    return am1 * e > tau;
  };
  // kept pages in page order: warp w owns pages [w seg, (w + 1) seg)
  const int seg = (((n + kSelWarps - 1) / kSelWarps) + 31) & ~31;
  const int p0 = warp * seg, p1 = min(n, p0 + seg);
  int mine = 0;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    mine += __popc(__ballot_sync(kFull, p < p1 && keep_of(p)));
  }
  if (lane == 0) s_cnt[warp] = mine;
  __syncthreads();
  int off = 0, total = 0;
  for (int w = 0; w < kSelWarps; ++w) {
    if (w < warp) off += s_cnt[w];
    total += s_cnt[w];
  }
  int32_t* out = a.sel + row * a.sel_stride;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    const bool k = p < p1 && keep_of(p);
    const unsigned bal = __ballot_sync(kFull, k);
    if (k) out[off + __popc(bal & ((1u << lane) - 1u))] = p;
    off += __popc(bal);
  }
  if (tid == 0) a.cnt[row] = total;
}

int g_mom_smem[12][64];

template <typename T, int D, int kG>
sa_status launch_moments(const GaussArgs& a, dim3 grid, cudaStream_t s, int* attr) {
  if (!ensure_smem(gauss_moments_kernel<T, D, kG>, 0, attr)) return SA_ERR_CUDA;
  gauss_moments_kernel<T, D, kG><<<grid, kMomThreads, 0, s>>>(a);
  return launch_status();
}

template <typename T, int D>
sa_status launch_moments_g(const GaussArgs& a, dim3 grid, cudaStream_t s, int slot) {
  if (a.G <= 4) return launch_moments<T, D, 4>(a, grid, s, g_mom_smem[slot * 3 + 0]);
  if (a.G <= 8) return launch_moments<T, D, 8>(a, grid, s, g_mom_smem[slot * 3 + 1]);
  return launch_moments<T, D, 16>(a, grid, s, g_mom_smem[slot * 3 + 2]);
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_gauss_select(const sa_cache* cache, const sa_batch* batch, const void* q,
                                     int32_t num_q_heads, float alpha, float scale, float* moments,
                                     int32_t max_pages, int32_t* sel_idx, int32_t* sel_cnt,
                                     int32_t sel_stride, float* tau_hat, int32_t* dev_status,
                                     void* stream) {
  using namespace sa;
  sa_status st = check_cache(cache, false, true);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (!cache->kstd || !q || !moments || !sel_idx || !sel_cnt) return SA_ERR_INVALID_ARG;
  if (max_pages <= 0 || max_pages < batch->bt_stride || sel_stride < max_pages) return SA_ERR_INVALID_ARG;
  if (!(alpha == 1.5f || alpha == 2.0f)) return SA_ERR_UNSUPPORTED;   // closed forms of the tail moments
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return SA_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  if (G > 16) return SA_ERR_UNSUPPORTED;
  if (int64_t(batch->batch) * num_q_heads * max_pages > (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
  GaussArgs a;
  a.meta = cache->meta; a.kstd = cache->kstd; a.q = q; a.bt = batch->block_table;
  a.seq_lens = batch->seq_lens; a.mom = reinterpret_cast<float2*>(moments); a.sel = sel_idx;
  a.cnt = sel_cnt; a.tau_hat = tau_hat; a.status = dev_status;
  a.H_kv = cache->num_kv_heads; a.H_q = num_q_heads; a.G = G; a.ps = cache->page_size;
  a.ps_shift = log2i(cache->page_size); a.num_blocks = cache->num_blocks;
  a.bt_stride = batch->bt_stride; a.max_pages = max_pages; a.sel_stride = sel_stride;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf(float(cache->head_dim));
  a.alpha = alpha;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 mgrid(unsigned((max_pages + kMomThreads - 1) / kMomThreads), unsigned(cache->num_kv_heads),
                   unsigned(batch->batch));
  const bool bf = cache->dtype == SA_BF16;
  if (cache->head_dim == 128)
    st = bf ? launch_moments_g<__nv_bfloat16, 128>(a, mgrid, s, 0) : launch_moments_g<__half, 128>(a, mgrid, s, 1);
  else
    st = bf ? launch_moments_g<__nv_bfloat16, 64>(a, mgrid, s, 2) : launch_moments_g<__half, 64>(a, mgrid, s, 3);
  if (st != SA_OK) return st;
  static int g_sel_smem[64];
  const int est_bytes = max_pages * int(sizeof(float));
  a.est_in_smem = est_bytes <= 160 * 1024;
  const int smem = a.est_in_smem ? est_bytes : 0;
  if (!ensure_smem(gauss_select_kernel, smem, g_sel_smem)) return SA_ERR_CUDA;
  gauss_select_kernel<<<dim3(unsigned(num_q_heads), unsigned(batch->batch)), kSelThreads, smem, s>>>(a);
  return launch_status();
}
