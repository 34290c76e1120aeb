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
//  (1) the page moments. With the page's dimensions taken as independent, a
//      query head's scores z = scale q . k on page p have
//        m_p = scale sum_d q_d mean_pd,  v_p = scale^2 sum_d q_d^2 std_pd^2,
//      for the G heads of a KV head a small dense product over the pages.
//      bf16 caches (gauss_moments_mma_kernel): on the tensor cores, with the
//      squares split exactly into two bf16 terms (a bf16 has 8 significant
//      bits, its square at most 16: hi = round(x^2), lo = x^2 - hi, both
//      bf16), so v = sum (qh + ql)(sh + sl) is four products of bf16 values,
//      each exact in float32, accumulated in float32 like m = sum q mean.
//      Persistent CTAs, one producer warp gathering each page's mean and std
//      rows by bulk copies into a shared-memory ring, four consumer warps of
//      8 pages each, the query fragments in registers. fp16 caches
//      (gauss_moments_kernel): one thread per page in float32 FMAs (the square
//      of an fp16 value can leave fp16's range, so it is not split).
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
  int B, H_kv, H_q, G, ps, ps_shift, num_blocks, bt_stride, max_pages, sel_stride;
  int est_in_smem;       // the selection kernel keeps every page's estimate in shared memory
  float scale, alpha;
};

template <typename T, int D, int kG>
__global__ void __launch_bounds__(kMomThreads) gauss_moments_kernel(GaussArgs a) {
  using E = Elem<T>;
  __shared__ float4 s_q[kG][D / 4];      // scale * q
  const int h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int G = a.G;
  pdl_wait();                            // everything the previous kernel wrote is visible
  pdl_trigger();
  const uint16_t* qb = static_cast<const uint16_t*>(a.q) + (int64_t(b) * a.H_q + int64_t(h) * G) * D;
  for (int i = tid; i < G * D; i += kMomThreads) {
    reinterpret_cast<float*>(s_q)[i] = a.scale * E::lo(uint32_t(qb[i]));
  }
  __syncthreads();
  const int L = a.seq_lens[b];
  const int n = min(L > 0 ? (L + a.ps - 1) >> a.ps_shift : 0, a.bt_stride);   // max_pages >= bt_stride
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

// ---------------------------------------------------------------------------
// bf16 page moments on the tensor cores
// ---------------------------------------------------------------------------
#ifndef SA_GMOM_MINB
#define SA_GMOM_MINB 1
#endif
#ifndef SA_GMOM_GROUPS
#define SA_GMOM_GROUPS 2
#endif
constexpr int kMmaWarps = 4;
constexpr int kMmaGroups = SA_GMOM_GROUPS;                 // 8-page groups per warp

// x * x rounded to bf16, per half, and the exact remainder x * x - round(x * x)
__device__ __forceinline__ void bf16x2_square_split(uint32_t x, uint32_t& hi, uint32_t& lo) {
  asm("mul.rn.bf16x2 %0, %1, %1;" : "=r"(hi) : "r"(x));
  asm("fma.rn.bf16x2 %0, %1, %1, %2;" : "=r"(lo) : "r"(x), "r"(hi ^ 0x80008000u));
}

// One warp per run of kMmaGroups groups of 8 pages of one (request, KV head);
// per group m16n8k16 products with the 8 pages as the n columns. The sum over
// k may take the dimensions in any order, so each lane reads its page's rows
// directly in 16-byte pieces: lane (g4, t4) loads, of page g4 of the group,
// the pieces at byte offsets 64 i + 16 t4 of the mean and std rows (the four
// lanes of a page read 64 contiguous bytes per load step), and piece i fills
// its B fragments of k steps 2 i (first 4 dimensions) and 2 i + 1 (next 4);
// q's A fragments, built once per warp, take the same order. A rows: kG <= 8:
// row g holds q_g and q_g^2 hi, row g + 8 zero and q_g^2 lo; kG == 16: rows g
// and g + 8 are heads g and g + 8, q^2 hi and lo in two tiles. The C
// fragment gives lane (g4, t4) head g4 (and g4 + 8) at pages 2 t4, 2 t4 + 1.
template <int D, int kG>
__global__ void __launch_bounds__(32 * kMmaWarps, SA_GMOM_MINB) gauss_moments_mma_kernel(GaussArgs a) {
  using E = Elem<__nv_bfloat16>;
  constexpr int NP = D / 32;                               // pieces per lane per row
  constexpr int KS = D / 16;                               // k steps
  constexpr int kTiles = kG > 8 ? 2 : 1;
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g4 = lane >> 2, t4 = lane & 3;
  pdl_wait();                                              // everything the previous kernel wrote is visible
  pdl_trigger();
  const int L = a.seq_lens[b];
  const int n_all = L > 0 ? (L + a.ps - 1) >> a.ps_shift : 0;
  if (n_all > a.bt_stride && blockIdx.x == 0 && h == 0 && threadIdx.x == 0) flag(a.status, SA_DEV_OVERFLOW);
  const int n = min(n_all, a.bt_stride);                   // max_pages >= bt_stride
  const int base = (blockIdx.x * kMmaWarps + warp) * (8 * kMmaGroups);
  if (base >= n) return;

  // block ids of every group (lane g4 of a quad: page g4)
  int blk[kMmaGroups];
#pragma unroll
  for (int gi = 0; gi < kMmaGroups; ++gi) {
    const int p = base + 8 * gi + g4;
    blk[gi] = p < n ? a.bt[int64_t(b) * a.bt_stride + p] : -1;
  }
  // q fragments in the pieces' k order
  uint32_t am[KS][4], av[kTiles][KS][4];
  {
    const uint4* q4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                     (int64_t(b) * a.H_q + int64_t(h) * a.G) * D);
    const bool r0 = g4 < a.G, r1 = kG > 8 && g4 + 8 < a.G;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const uint4 u0 = r0 ? q4[(g4 * D) / 8 + 4 * i + t4] : z;
      const uint4 u1 = r1 ? q4[((g4 + 8) * D) / 8 + 4 * i + t4] : z;
      const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w}, w1[4] = {u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int kk = 2 * i + hf;
        uint32_t h0, l0, h2, l2;
        bf16x2_square_split(w0[2 * hf], h0, l0);
        bf16x2_square_split(w0[2 * hf + 1], h2, l2);
        am[kk][0] = w0[2 * hf]; am[kk][2] = w0[2 * hf + 1];
        if constexpr (kG > 8) {
          uint32_t h1, l1, h3, l3;
          bf16x2_square_split(w1[2 * hf], h1, l1);
          bf16x2_square_split(w1[2 * hf + 1], h3, l3);
          am[kk][1] = w1[2 * hf]; am[kk][3] = w1[2 * hf + 1];
          av[0][kk][0] = h0; av[0][kk][1] = h1; av[0][kk][2] = h2; av[0][kk][3] = h3;
          av[kTiles - 1][kk][0] = l0; av[kTiles - 1][kk][1] = l1;
          av[kTiles - 1][kk][2] = l2; av[kTiles - 1][kk][3] = l3;
        } else {
          am[kk][1] = 0u; am[kk][3] = 0u;
          av[0][kk][0] = h0; av[0][kk][1] = l0; av[0][kk][2] = h2; av[0][kk][3] = l2;
        }
      }
    }
  }
  const uint4* meta4 = static_cast<const uint4*>(a.meta);
  const uint4* std4 = static_cast<const uint4*>(a.kstd);
  auto good = [&](int bk) { return bk >= 0 && bk < a.num_blocks; };
  auto load = [&](int bk, uint4 (&pm)[NP], uint4 (&pv)[NP]) {
    const int64_t ph = int64_t(bk) * a.H_kv + h;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      pm[i] = good(bk) ? __ldg(meta4 + (ph * 3 + 2) * (D / 8) + 4 * i + t4) : make_uint4(0u, 0u, 0u, 0u);
      pv[i] = good(bk) ? __ldg(std4 + ph * (D / 8) + 4 * i + t4) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  const float sc = a.scale, sc2 = a.scale * a.scale;
  uint4 cm_[NP], cs_[NP];
  load(blk[0], cm_, cs_);
#pragma unroll
  for (int gi = 0; gi < kMmaGroups; ++gi) {
    const int p0 = base + 8 * gi;
    if (p0 >= n) break;
    uint4 nm[NP], ns[NP];
    if (gi + 1 < kMmaGroups) load(blk[gi + 1], nm, ns);    // the next group's rows in flight
    const int pl = p0 + g4;
    if (pl < n && !good(blk[gi]) && t4 == 0) flag(a.status, SA_DEV_BAD_BLOCK);
    const uint32_t ok = __ballot_sync(kFull, good(blk[gi]));
    float cm[4] = {0.f, 0.f, 0.f, 0.f}, cv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const uint32_t wm[4] = {cm_[i].x, cm_[i].y, cm_[i].z, cm_[i].w};
      const uint32_t ws[4] = {cs_[i].x, cs_[i].y, cs_[i].z, cs_[i].w};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int kk = 2 * i + hf;
        uint32_t sh0, sl0, sh1, sl1;
        bf16x2_square_split(ws[2 * hf], sh0, sl0);
        bf16x2_square_split(ws[2 * hf + 1], sh1, sl1);
        E::mma(cm, am[kk], wm[2 * hf], wm[2 * hf + 1]);
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
          E::mma(cv, av[t][kk], sh0, sh1);
          E::mma(cv, av[t][kk], sl0, sl1);
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < kTiles; ++hh) {
      const int g = g4 + 8 * hh;
      if (g >= a.G) continue;
      float2* out = a.mom + (int64_t(b) * a.H_q + int64_t(h) * a.G + g) * a.max_pages + p0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 2 * t4 + e;
        if (p0 + j >= n) continue;
        const float m = kG > 8 ? cm[2 * hh + e] : cm[e];
        const float v = kG > 8 ? cv[2 * hh + e] : cv[e] + cv[2 + e];
        out[j] = ((ok >> (4 * j)) & 1u) ? make_float2(sc * m, sc2 * v) : make_float2(-INFINITY, 0.f);
      }
    }
    if (gi + 1 < kMmaGroups) {
#pragma unroll
      for (int i = 0; i < NP; ++i) { cm_[i] = nm[i]; cs_[i] = ns[i]; }
    }
  }
}

// s += x with the rounding error carried in c (Kahan-Babuska-Neumaier)
__device__ __forceinline__ void csum(float& s, float& c, float x) {
  const float t = s + x;
  c += fabsf(s) >= fabsf(x) ? (s - t) + x : (x - t) + s;
  s = t;
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

// a + b = s + e exactly (Knuth's TwoSum)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// a compensated pair (s, c) summed over the warp, the rounding of each step kept in c
__device__ __forceinline__ void warp_sum_pair(float& s, float& c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(kFull, s, o), c2 = __shfl_xor_sync(kFull, c, o);
    float t, e;
    two_sum(s, s2, t, e);
    s = t;
    c = c + c2 + e;
  }
}

constexpr int kSelBatch = 16;                              // page moments in flight per thread

__global__ void __launch_bounds__(kSelThreads) gauss_select_kernel(GaussArgs a) {
  __shared__ float s_red[kSelWarps][4];                    // per warp: S1 (s, c), S2 (s, c)
  __shared__ int s_n[kSelWarps];
  __shared__ int s_cnt[kSelWarps];
  __shared__ float s_par[4];                               // mu_a, s_a, N, closed-form tau
  __shared__ int s_mode;                                   // 0 no tokens, 1 closed form, 2 solve
  __shared__ float s_tau;
  const int gq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  pdl_wait();                                              // the moments are complete
  pdl_trigger();
  const int L = a.seq_lens[b];
  const int n_all = L > 0 ? (L + a.ps - 1) >> a.ps_shift : 0;
  if (n_all > a.bt_stride && tid == 0) flag(a.status, SA_DEV_OVERFLOW);
  const int n = min(n_all, a.bt_stride);                    // max_pages >= bt_stride
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
  int f_s = 0;
  float s1 = 0.f, c1 = 0.f, s2 = 0.f, c2 = 0.f;
  for (int p0 = tid; p0 < n; p0 += kSelBatch * kSelThreads) {
    float2 mv[kSelBatch];
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u) {                   // every load issued before any is used
      const int p = p0 + u * kSelThreads;
      mv[u] = p < n ? __ldcg(mom + p) : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u) {
      const int p = p0 + u * kSelThreads;
      const bool ok = p < n && mv[u].x > -INFINITY && mv[u].x < INFINITY;
      const int fi = min(a.ps, L - (p << a.ps_shift));
      if (cached && p < n) s_est[p] = ok ? est_max(mv[u], fi, a.ps, kappa_full) : -INFINITY;
      if (!ok) continue;
      const float f = float(fi);
      f_s += fi;
      csum(s1, c1, f * mv[u].x);
      csum(s2, c2, f * (mv[u].y + mv[u].x * mv[u].x));
    }
  }
  f_s = __reduce_add_sync(kFull, f_s);
  warp_sum_pair(s1, c1);
  warp_sum_pair(s2, c2);
  if (lane == 0) {
    s_n[warp] = f_s;
    s_red[warp][0] = s1; s_red[warp][1] = c1; s_red[warp][2] = s2; s_red[warp][3] = c2;
  }
  __syncthreads();
  const bool sparsemax = a.alpha == 2.0f;
  if (tid == 0) {                                           // float64 on one thread only
    long long N = 0;
    double S1 = 0.0, S2 = 0.0;
    for (int w = 0; w < kSelWarps; ++w) {
      N += s_n[w];
      S1 += double(s_red[w][0]) + double(s_red[w][1]);
      S2 += double(s_red[w][2]) + double(s_red[w][3]);
    }
    int mode = 0;                                           // nothing resolves: only the tail
    if (N > 0) {
      const double Nd = double(N), Md = S1 / Nd;
      const float M = float(Md), V = float(fmax(S2 / Nd - Md * Md, 0.0));
      const float am1 = a.alpha - 1.0f;
      const float mu_a = am1 * M, s_a = am1 * sqrtf(V), Nf = float(Nd);
      s_par[0] = mu_a; s_par[1] = s_a; s_par[2] = Nf;
      s_par[3] = mu_a - (sparsemax ? 1.0f / Nf : rsqrtf(Nf));   // N (mu_a - tau)^r = 1 when s_a = 0
      mode = s_a <= 0.f ? 1 : 2;
    }
    s_mode = mode;
  }
  __syncthreads();
  const int mode = s_mode;
  float tau = mode == 1 ? s_par[3] : -INFINITY;
  if (mode == 2) {
    // the constraint at kSelThreads points from (alpha - 1) M - 1 (left of the
    // root by Jensen) to 10 deviations above the mean, one per thread; Newton
    // starts from the largest point still left of the root (any start there
    // converges monotonically: the function is convex and decreasing)
    const float mu_a = s_par[0], s_a = s_par[1], Nf = s_par[2];
    const float lo = mu_a - 1.0f, span = 1.0f + 10.0f * s_a;
    auto point = [&](int i) { return lo + span * (float(i) / float(kSelThreads)); };
    float e, de;
    tail_moment(mu_a, s_a, point(tid), sparsemax, e, de);
    const unsigned pos = __ballot_sync(kFull, Nf * e - 1.0f > 0.f);
    if (lane == 0) s_cnt[warp] = pos ? warp * 32 + 31 - __clz(pos) : -1;
    __syncthreads();
    if (tid == 0) {
      int best = 0;
      for (int w = 0; w < kSelWarps; ++w) best = max(best, s_cnt[w]);
      tau = point(best);
      for (int it = 0; it < 100; ++it) {
        tail_moment(mu_a, s_a, tau, sparsemax, e, de);
        const float g = Nf * e - 1.0f;
        if (!(g > 0.f) || !(de < 0.f)) break;
        const float step = -g / (Nf * de);
        tau += step;
        if (step <= 1e-7f * (1.0f + fabsf(tau))) break;
      }
    }
  }
  if (tid == 0) {
    s_tau = tau;
    if (a.tau_hat) a.tau_hat[row] = tau;
  }
  __syncthreads();
  tau = s_tau;
  const float am1 = a.alpha - 1.0f;
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
#pragma unroll 4
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
#pragma unroll 4
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
  return launch_ex(gauss_moments_kernel<T, D, kG>, grid, dim3(kMomThreads), 0, s, true, 1u, a) == cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

template <int D>
sa_status launch_moments_mma(const GaussArgs& a, dim3 grid, cudaStream_t s) {
  const cudaError_t e = a.G <= 8 ? launch_ex(gauss_moments_mma_kernel<D, 8>, grid, dim3(32 * kMmaWarps), 0, s, true, 1u, a)
                                  : launch_ex(gauss_moments_mma_kernel<D, 16>, grid, dim3(32 * kMmaWarps), 0, s, true, 1u, a);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
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
  if (!aligned16(q)) return SA_ERR_INVALID_ARG;
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
  a.B = batch->batch; a.H_kv = cache->num_kv_heads; a.H_q = num_q_heads; a.G = G; a.ps = cache->page_size;
  a.ps_shift = log2i(cache->page_size); a.num_blocks = cache->num_blocks;
  a.bt_stride = batch->bt_stride; a.max_pages = max_pages; a.sel_stride = sel_stride;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf(float(cache->head_dim));
  a.alpha = alpha;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = cache->dtype == SA_BF16;
  if (bf) {
    const int per_cta = 8 * kMmaGroups * kMmaWarps;
    const dim3 grid(unsigned((batch->bt_stride + per_cta - 1) / per_cta), unsigned(cache->num_kv_heads),
                    unsigned(batch->batch));
    st = cache->head_dim == 128 ? launch_moments_mma<128>(a, grid, s) : launch_moments_mma<64>(a, grid, s);
  } else {
    const dim3 mgrid(unsigned((batch->bt_stride + kMomThreads - 1) / kMomThreads), unsigned(cache->num_kv_heads),
                     unsigned(batch->batch));
    st = cache->head_dim == 128 ? launch_moments_g<__half, 128>(a, mgrid, s, 1) : launch_moments_g<__half, 64>(a, mgrid, s, 3);
  }
  if (st != SA_OK) return st;
  static int g_sel_smem[64];
  const int est_bytes = max_pages * int(sizeof(float));
  a.est_in_smem = est_bytes <= 160 * 1024;
  const int smem = a.est_in_smem ? est_bytes : 0;
  if (!ensure_smem(gauss_select_kernel, smem, g_sel_smem)) return SA_ERR_CUDA;
  // both launches programmatic: each kernel waits on the device for its
  // predecessor before reading anything, so only the launch latency overlaps
  return launch_ex(gauss_select_kernel, dim3(unsigned(num_q_heads), unsigned(batch->batch)), dim3(kSelThreads),
                   size_t(smem), s, true, 1u, a) == cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}
