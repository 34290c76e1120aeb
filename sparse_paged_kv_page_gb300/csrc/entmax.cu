// sa_sparse_decode_entmax: attention over the selected pages with alpha-entmax
// in place of the softmax.
//
// "EntmaxKV" README, "How it works" and "Quick start": the selected pages are
// attended exactly, the normaliser being alpha-entmax (alpha = 1.5 by
// default; 1.5 and 2 have closed forms): with a_j = (alpha - 1) z_j, z_j the
// scaled logits of the selection, p_j = (a_j - tau)_+ ^ (1 / (alpha - 1)) and
// tau fixed by sum_j p_j = 1.
//
// Three launches, chained by programmatic dependent launch:
//  (1) the decode kernel in its logits-only mode writes z for every selected
//      token (K is read; V is not);
//  (2) entmax_tau_kernel, one CTA per (request, query head), finds tau:
//      only entries above a_max - 1 can ever be in the support (tau >= a_max
//      - 1): the CTA gathers those. For alpha = 2 and 1.5 it ranks them and
//      takes the closed-form root of the largest support whose root stays
//      below its smallest member (the sort-based rule, exact); for
//      other alpha one warp runs Newton's method from a_max - 1, which rises
//      monotonically to the root of the convex, decreasing f(tau) = sum_j
//      (a_j - tau)_+^r - 1 (r = 1 / (alpha - 1) >= 1), with the closed-form
//      shortcut of each iterate's support where one exists. float32;
//  (3) entmax_attend_kernel, split over tokens, one CTA per (split, request,
//      KV head): each warp tests 32 tokens at a time against the G heads' tau
//      and loads V rows only for tokens some head of the group keeps
//      (entmax is sparse), accumulating sum_j p_j v_j and sum_j p_j in fp32;
//      the splits of a (request, KV head), at most 8, form a thread-block
//      cluster: each stores its partials into the shared memory of the CTA
//      that adds that slice, which adds them in split order (where a cluster
//      cannot launch, the last CTA adds them from the workspace), dividing
//      by sum_j p_j (1 up to the rounding of tau).
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {


constexpr int kThreads = 256;
constexpr int kMaxClusterSplits = 8;     // splits of a unit merged inside one (portable) cluster
constexpr int kWarps = kThreads / 32;
// Dynamic shared memory of the weighted-V kernel: the warps' partials
// ([kWarps][G][D + 1] floats), the (block, fill) entries, and the cluster
// merge's receive area (every peer's partial of this CTA's slice,
// [nsplit][chunk] <= G * D + kMaxClusterSplits floats, and every peer's
// sum p of each row, [kMaxClusterSplits][16]).
inline int64_t attend_smem(int G, int D, int ent_cap) {
  return int64_t(kWarps) * G * (D + 1) * 4 + int64_t(ent_cap) * 8 +
         (int64_t(G) * D + kMaxClusterSplits + kMaxClusterSplits * 16) * 4;
}
constexpr int kCand = 256;               // candidates each warp of the tau kernel gathers (beyond: the row is streamed)
constexpr int kMaxIter = 100;
constexpr int kRowReg = 16;              // row entries per thread the tau kernel keeps in registers
constexpr int kSortMax = kWarps * kCand; // every gathered candidate can be ranked
constexpr int kRankDirect = 128;         // up to this many candidates: rank by direct counting
constexpr int kPrefilterRounds = 3;      // Newton rounds that thin a larger candidate set first
static_assert(kCand == 256, "the per-warp sort holds 8 candidates a lane");

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
  int32_t* tickets;      // [B, H_kv]: splits of the (request, KV head) done
  void* out;
  int32_t* status;
  int H_kv, H_q, G, ps, ps_shift, num_blocks, bt_stride, sel_stride, logits_stride, nsplit, ent_cap;
  int H_u, kv_div;       // selection units per request (H_kv, or H_q per query head) and per KV head
  float alpha;
};

// 0: generic alpha (Newton only), 1: alpha = 1.5, 2: alpha = 2
__host__ __device__ inline int alpha_kind(float alpha) {
  return alpha == 2.0f ? 2 : (alpha == 1.5f ? 1 : 0);
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

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// s += x with the rounding error carried in c (Kahan-Babuska-Neumaier)
__device__ __forceinline__ void csum(float& s, float& c, float x) {
  const float t = s + x;
  c += fabsf(s) >= fabsf(x) ? (s - t) + x : (x - t) + s;
  s = t;
}

// The support sums at tau over this lane's share of the entries: count,
// sum d^r, sum d^(r-1), min d over the members (d = a - tau > 0) and max d
// over the others.
struct Sums {
  float k, p0, p1, mn, mo;
};

__device__ __forceinline__ void add_entry(float x, float tau, int kind, float r, Sums& s, float& c0,
                                          float& c1) {
  const float d = x - tau;
  if (d > 0.f) {
    s.k += 1.f;
    if (kind == 2) {
      csum(s.p0, c0, d);
      s.p1 += 1.f;
    } else if (kind == 1) {
      csum(s.p0, c0, d * d);
      csum(s.p1, c1, d);
    } else {
      const float t = powf(d, r - 1.f);
      csum(s.p0, c0, t * d);
      csum(s.p1, c1, t);
    }
    s.mn = fminf(s.mn, d);
  } else {
    s.mo = fmaxf(s.mo, d);
  }
}

// One Newton round given the warp's reduced sums: returns true when tau is final.
__device__ __forceinline__ bool newton_round(const Sums& s, int kind, float r, float& tau) {
  if (s.k <= 0.f) return true;                              // (cannot happen below the root)
  const float f = s.p0 - 1.f;
  if (kind != 0) {
    // closed-form root of this support, as an offset from tau, without
    // cancellation: alpha 2: sum d = 1 + k delta; alpha 1.5: the smaller root
    // of k delta^2 - 2 delta sum d + sum d^2 - 1 = 0
    const float delta = kind == 2 ? f / s.k : f / (s.p1 + sqrtf(fmaxf(s.p1 * s.p1 - s.k * f, 0.f)));
    if (delta >= s.mo && delta < s.mn) {
      // every member stays above tau + delta and every other entry at or
      // below it: the support is consistent with its root. A large step came
      // from sums taken far from the root (d near 1), so take one more round
      tau += delta;
      return fabsf(delta) <= 1e-6f * (1.f + fabsf(tau));
    }
  }
  if (f <= 0.f) return true;                                // at the root up to rounding
  const float step = f / (r * s.p1);
  if (step <= 1e-7f * fmaxf(1.f, fabsf(tau))) return true;
  tau += step;
  return false;
}

// a = (alpha - 1) z, non-finite logits never entering
__device__ __forceinline__ float a_of(float z, float am1) {
  return (z > -INFINITY && z < INFINITY) ? am1 * z : -INFINITY;
}

// One warp's Newton rounds over the candidates gathered per warp
// (cand[w][0, cnt[w])); every lane returns tau.
__device__ float solve_gathered(const float (*cand)[kCand], const int* cnt, float tau, int kind,
                                float r) {
  const int lane = threadIdx.x & 31;
  for (int it = 0; it < kMaxIter; ++it) {
    Sums s = {0.f, 0.f, 0.f, INFINITY, -INFINITY};
    float c0 = 0.f, c1 = 0.f;
    for (int w = 0; w < kWarps; ++w)
      for (int j = lane; j < cnt[w]; j += 32) add_entry(cand[w][j], tau, kind, r, s, c0, c1);
    s.p0 += c0;
    s.p1 += c1;
    s.k = warp_sum_f(s.k); s.p0 = warp_sum_f(s.p0); s.p1 = warp_sum_f(s.p1);
    s.mn = warp_min_f(s.mn); s.mo = warp_max_f(s.mo);
    if (newton_round(s, kind, r, tau)) break;
  }
  return tau;
}

// All threads over the whole row (entries <= skip never in the support), the
// sums combined through shared memory; every thread returns the same tau.
__device__ float solve_row(const float* z, int n, float am1, float tau, float skip, int kind, float r,
                           float (*red)[kWarps][5]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int it = 0; it < kMaxIter; ++it) {
    Sums s = {0.f, 0.f, 0.f, INFINITY, -INFINITY};
    float c0 = 0.f, c1 = 0.f;
    for (int j = threadIdx.x; j < n; j += kThreads) {
      const float x = a_of(__ldcg(z + j), am1);
      if (x > skip) add_entry(x, tau, kind, r, s, c0, c1);
    }
    s.p0 += c0;
    s.p1 += c1;
    s.k = warp_sum_f(s.k); s.p0 = warp_sum_f(s.p0); s.p1 = warp_sum_f(s.p1);
    s.mn = warp_min_f(s.mn); s.mo = warp_max_f(s.mo);
    float(*rb)[5] = red[it & 1];                            // alternate buffers: one barrier a round
    if (lane == 0) {
      rb[warp][0] = s.k; rb[warp][1] = s.p0; rb[warp][2] = s.p1; rb[warp][3] = s.mn; rb[warp][4] = s.mo;
    }
    __syncthreads();
    s = {rb[0][0], rb[0][1], rb[0][2], rb[0][3], rb[0][4]};
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      s.k += rb[w][0]; s.p0 += rb[w][1]; s.p1 += rb[w][2]; s.mn = fminf(s.mn, rb[w][3]);
      s.mo = fmaxf(s.mo, rb[w][4]);
    }
    if (newton_round(s, kind, r, tau)) break;
  }
  return tau;
}

// One warp sorts 256 values descending, 8 per lane in blocked order (lane l
// holds entries 8 l .. 8 l + 7): the bitonic network, pairs (e, e ^ j) inside
// a lane swapped in registers, across lanes exchanged by shuffle. The stage
// loops stay rolled: the code runs once per CTA, so its size is its cost.
template <int J>
__device__ __forceinline__ void bitonic_in_lane(float (&v)[8], int lane, int k) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if ((i & J) == 0) {
      const bool desc = ((lane * 8 + i) & k) == 0;
      const float x = v[i], y = v[i | J];
      v[i] = desc ? fmaxf(x, y) : fminf(x, y);
      v[i | J] = desc ? fminf(x, y) : fmaxf(x, y);
    }
  }
}

__device__ void warp_sort256_desc(float (&v)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int k = 2; k <= 256; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j >= 8; j >>= 1) {
      const int lj = j >> 3;
      const bool lower = (lane & lj) == 0;                  // the smaller index of the pair
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = __shfl_xor_sync(kFull, v[i], lj);
        const bool desc = ((lane * 8 + i) & k) == 0;
        v[i] = (lower == desc) ? fmaxf(v[i], o) : fminf(v[i], o);
      }
    }
    if (k >= 8) bitonic_in_lane<4>(v, lane, k);
    if (k >= 4) bitonic_in_lane<2>(v, lane, k);
    bitonic_in_lane<1>(v, lane, k);
  }
}

// entries of the descending run r[0, n) that are >= x (ge) or > x (!ge)
__device__ __forceinline__ int count_above(const float* r, int n, float x, bool ge) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const float y = r[mid];
    if (ge ? (y >= x) : (y > x)) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// alpha 1.5 / 2, one warp: the candidates sorted descending in srt[0, m),
// centred on their maximum (x' = a - a_max <= 0). With S1, S2 the sums of
// x' and x'^2 over the k largest, the root of that support is
//   alpha 2:   t_k = (S1 - 1) / k
//   alpha 1.5: t_k = (S1 - sqrt(S1^2 - k S2 + k)) / k   (k t^2 - 2 t S1 + S2 - 1 = 0,
//              the smaller root; both terms <= 0, so nothing cancels)
// and the support is the largest k with t_k below its k-th value. Returns
// that t_k (in the centred units); every lane returns it.
__device__ float tau_sorted(const float* srt, int m, int kind) {
  const int lane = threadIdx.x & 31;
  const int per = (m + 31) >> 5;
  const int j0 = min(m, lane * per), j1 = min(m, j0 + per);
  float s1 = 0.f, s2 = 0.f;
  for (int j = j0; j < j1; ++j) {
    const float x = srt[j];
    s1 += x;
    s2 = fmaf(x, x, s2);
  }
  // exclusive prefix over the lanes
  float e1 = s1, e2 = s2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y1 = __shfl_up_sync(kFull, e1, o), y2 = __shfl_up_sync(kFull, e2, o);
    if (lane >= o) { e1 += y1; e2 += y2; }
  }
  e1 -= s1;
  e2 -= s2;
  int best = 0;
  float tbest = 0.f;
  for (int j = j0; j < j1; ++j) {
    const float x = srt[j];
    e1 += x;
    e2 = fmaf(x, x, e2);
    const float k = float(j + 1);
    const float t = kind == 2 ? (e1 - 1.f) / k : (e1 - sqrtf(fmaxf(fmaf(e1, e1, k - k * e2), 0.f))) / k;
    if (t < x) { best = j + 1; tbest = t; }
  }
  int kmax = best;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
  const unsigned who = __ballot_sync(kFull, best == kmax);
  return __shfl_sync(kFull, tbest, __ffs(who) - 1);
}

// tau of one (request, query head). The CTA reads the row once into registers
// (rows up to kThreads * kRowReg entries; longer rows are read again from L2)
// for its maximum, gathers the entries above maximum - 1 per warp, and then,
// for alpha 1.5 / 2, ranks them (a few: by counting; more: a sort per warp and
// a merge of the runs by binary search) and takes the closed form of the
// largest consistent support; generic alpha iterates Newton's method instead.
__global__ void __launch_bounds__(kThreads) entmax_tau_kernel(EntArgs a) {
  __shared__ float s_c[kWarps][kCand];
  __shared__ float s_srt[kSortMax];
  __shared__ int s_n[kWarps];
  __shared__ float red[2][kWarps][5];
  __shared__ float s_mx[kWarps];
  const int gq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  pdl_trigger();                                          // the weighted-V kernel may start its prologue
  pdl_wait();                                             // the logits of this call are written
  int c = a.cnt[b * a.H_u + gq / a.G];
  c = max(0, min(c, a.sel_stride));
  const int n = c << a.ps_shift;
  const float* z = a.logits + (int64_t(b) * a.H_q + gq) * a.logits_stride;
  const float am1 = a.alpha - 1.0f;
  const bool in_reg = n <= kThreads * kRowReg;
  float xr[kRowReg];
  float mx = -INFINITY;
  if (in_reg) {
#pragma unroll
    for (int i = 0; i < kRowReg; ++i) {
      const int j = i * kThreads + tid;
      xr[i] = j < n ? a_of(__ldcg(z + j), am1) : -INFINITY;
      mx = fmaxf(mx, xr[i]);
    }
  } else {
#pragma unroll 4
    for (int j = tid; j < n; j += kThreads) mx = fmaxf(mx, a_of(__ldcg(z + j), am1));
  }
  mx = warp_max_f(mx);
  if (lane == 0) s_mx[warp] = mx;
  __syncthreads();
  mx = s_mx[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, s_mx[w]);
  const int64_t row = int64_t(b) * a.H_q + gq;
  float tau = __int_as_float(0x7fc00000);                 // NaN: no finite logit
  if (mx > -INFINITY) {
    const int kind = alpha_kind(a.alpha);
    const float r = 1.0f / am1;
    // gather a > a_max - 1 (with a margin for the rounding of a_max - 1);
    // warp w takes entries i * kThreads + 32 w + lane, i ascending
    const float lo = (mx - 1.0f) - 1e-6f * (1.0f + fabsf(mx));
    int got = 0;
    auto gather = [&](float x) {
      const bool take = x > lo;
      const unsigned bal = __ballot_sync(kFull, take);
      const int pos = got + __popc(bal & ((1u << lane) - 1u));
      if (take && pos < kCand) s_c[warp][pos] = x;
      got += __popc(bal);
    };
    if (in_reg) {
#pragma unroll
      for (int i = 0; i < kRowReg; ++i) gather(xr[i]);
    } else {
      for (int j0 = 0; j0 < n; j0 += kThreads) {
        const int j = j0 + tid;
        gather(j < n ? a_of(__ldcg(z + j), am1) : -INFINITY);
      }
    }
    if (lane == 0) s_n[warp] = got;
    __syncthreads();
    int m = 0;
    bool fits = true;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) { m += s_n[w]; fits &= s_n[w] <= kCand; }
    if (!fits) {                                            // many near-equal logits
      tau = solve_row(z, n, am1, mx - 1.0f, lo, kind, r, red);
    } else if (kind == 0 || m > kSortMax) {
      if (warp != 0) return;
      tau = solve_gathered(s_c, s_n, mx - 1.0f, kind, r);
    } else {
      if (m > kRankDirect) {
        // Shrink the set first: Newton's method from a_max - 1 stays left of
        // the root, so after a few rounds every support member still lies
        // above the iterate (less a margin for float32 rounding) and the
        // entries at or below it can be dropped.
        if (warp == 0) {
          float t = mx - 1.0f;
          for (int it = 0; it < kPrefilterRounds; ++it) {
            Sums su = {0.f, 0.f, 0.f, INFINITY, -INFINITY};
            float c0 = 0.f, c1 = 0.f;
            for (int w = 0; w < kWarps; ++w)
              for (int j = lane; j < s_n[w]; j += 32) add_entry(s_c[w][j], t, kind, r, su, c0, c1);
            su.p0 = warp_sum_f(su.p0 + c0);
            su.p1 = warp_sum_f(su.p1 + c1);
            const float f = su.p0 - 1.f;
            if (!(f > 0.f) || !(su.p1 > 0.f)) break;
            t += f / (r * su.p1);
          }
          if (lane == 0) s_mx[0] = t - 1e-4f * (1.f + fabsf(t));
        }
        __syncthreads();
        const float t_lo = s_mx[0];
        // each warp compacts its own run in place (order kept; writes never pass reads)
        const int nw = s_n[warp];
        int kept = 0;
        for (int j0 = 0; j0 < nw; j0 += 32) {
          const int j = j0 + lane;
          const float x = j < nw ? s_c[warp][j] : -INFINITY;
          const bool take = x > t_lo;
          const unsigned bal = __ballot_sync(kFull, take);
          __syncwarp();
          if (take) s_c[warp][kept + __popc(bal & ((1u << lane) - 1u))] = x;
          kept += __popc(bal);
          __syncwarp();
        }
        __syncthreads();                                    // every warp has read the old counts
        if (lane == 0) s_n[warp] = kept;
        __syncthreads();
        m = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) m += s_n[w];
      }
      if (m > kRankDirect) {
      // each warp sorts its own candidates, then an entry's rank is its place
      // in its run plus the entries above it in the other runs (ties: runs
      // in warp order), every rank distinct
      {
        float v[8];
        const int nw = s_n[warp];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = lane * 8 + i;
          v[i] = e < nw ? s_c[warp][e] : -INFINITY;
        }
        warp_sort256_desc(v);
#pragma unroll
        for (int i = 0; i < 8; ++i) s_c[warp][lane * 8 + i] = v[i];
      }
      __syncthreads();
      for (int ci = tid; ci < m; ci += kThreads) {
        int w = 0, off = 0;
        while (ci >= off + s_n[w]) off += s_n[w++];
        const int l = ci - off;
        const float x = s_c[w][l];
        int rank = l;
        for (int u = 0; u < kWarps; ++u)
          if (u != w) rank += count_above(s_c[u], s_n[u], x, u < w);
        s_srt[rank] = x - mx;
      }
      __syncthreads();
      if (warp != 0) return;
      tau = mx + tau_sorted(s_srt, m, kind);
      } else {
      // rank of each candidate among all: larger value first, ties by gather position
      for (int ci = tid; ci < m; ci += kThreads) {
        int w = 0, off = 0;
        while (ci >= off + s_n[w]) off += s_n[w++];
        const int gi = w * kCand + (ci - off);
        const float x = s_c[w][ci - off];
        int rank = 0;
        for (int v = 0; v < kWarps; ++v) {
          const int nv = s_n[v];
          for (int jj = 0; jj < nv; ++jj) {
            const float y = s_c[v][jj];
            rank += (y > x) | ((y == x) & (v * kCand + jj < gi));
          }
        }
        s_srt[rank] = x - mx;
      }
      __syncthreads();
      if (warp != 0) return;
      tau = mx + tau_sorted(s_srt, m, kind);
      }
    }
  }
  if (tid == 0) {
    a.tau[row] = tau;
    if (a.tau_out) a.tau_out[row] = tau;
  }
}

template <typename T, int D, int kG, bool kCluster>
__global__ void __launch_bounds__(kThreads, 2) entmax_attend_kernel(EntArgs a) {
  using E = Elem<T>;
  constexpr int DPL = D / 32;                              // dims per lane: 4 (D 128) or 2 (D 64)
  constexpr int kU = kG > 8 ? 4 : 8;                       // V rows in flight per warp
  extern __shared__ float4 smem_f4[];
  float* s_red = reinterpret_cast<float*>(smem_f4);       // [warps][G][D], then [warps][G]
  int2* s_ent = reinterpret_cast<int2*>(s_red + kWarps * a.G * (D + 1));
  __shared__ float s_tau[kG];
  __shared__ float s_l[kG];
  __shared__ int s_last;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = a.G;
  // Cluster merge: peers store into this CTA's receive area only after this
  // arrive has been waited on, i.e. once every CTA of the cluster has started.
  const bool push = kCluster && a.nsplit > 1;
  if (push) cluster_arrive_relaxed();
  // the selection and lengths come from before the logits pass: resolve the
  // entries this CTA touches to (block, fill) before waiting for the thresholds
  const int kvh = h / a.kv_div;                           // the unit's KV head
  int c = a.cnt[b * a.H_u + h];
  c = max(0, min(c, a.sel_stride));
  const int n = c << a.ps_shift;
  const int per = (((n + a.nsplit - 1) / a.nsplit) + 31) & ~31;
  const int t_lo = min(n, split * per), t_hi = min(n, t_lo + per);
  const int L = a.seq_lens[b];
  const int n_pages_req = L > 0 ? (L + a.ps - 1) >> a.ps_shift : 0;
  const int32_t* sel = a.sel + int64_t(b * a.H_u + h) * a.sel_stride;
  const int32_t* btb = a.bt + int64_t(b) * a.bt_stride;
  const int e_lo = t_lo >> a.ps_shift;
  const int e_n = t_hi > t_lo ? min(((t_hi - 1) >> a.ps_shift) - e_lo + 1, a.ent_cap) : 0;
  for (int i = tid; i < e_n; i += kThreads) {
    const int page = sel[e_lo + i];
    int blk = -1, fill = 0;
    if (page >= 0 && page < n_pages_req && page < a.bt_stride) {
      const int x = btb[page];
      if (x >= 0 && x < a.num_blocks) { blk = x; fill = min(a.ps, L - (page << a.ps_shift)); }
    }
    s_ent[i] = make_int2(blk, fill);
  }
  pdl_wait();                                              // the thresholds are written
  if (tid < G) s_tau[tid] = __ldcg(&a.tau[int64_t(b) * a.H_q + h * G + tid]);
  __syncthreads();

  const float am1 = a.alpha - 1.0f;
  const int kind = alpha_kind(a.alpha);
  const float r = 1.0f / am1;
  const float* zb = a.logits + (int64_t(b) * a.H_q + int64_t(h) * G) * a.logits_stride;

  float acc[kG][DPL], psum[kG];
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    psum[g] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[g][d] = 0.f;
  }
  const T* vbase = static_cast<const T*>(a.v);
  for (int base = t_lo + warp * 32; base < t_hi; base += kWarps * 32) {
    // p of token base + lane for every head of the group
    const int j = base + lane;
    float p[kG];
    bool keep = false;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      p[g] = 0.f;
      if (g < G && j < t_hi) {
        const float zz = __ldcg(zb + int64_t(g) * a.logits_stride + j);
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
          const T* vrow = vbase + ((int64_t(en.x) * a.H_kv + kvh) * a.ps + s) * D + lane * DPL;
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
      if (lane == 0) s_red[kWarps * G * D + warp * G + g] = ps;
    }
  }
  __syncthreads();
  const int64_t prow = (int64_t(b) * a.H_q + int64_t(h) * G) * a.nsplit;   // (b, head h*G, split 0)
  if (!kCluster && a.nsplit > 1) {                         // the ticket merge reads these
    for (int idx = tid; idx < G * D; idx += kThreads) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += s_red[w * G * D + idx];
      const int g = idx / D, d = idx % D;
      a.part_o[((prow + int64_t(g) * a.nsplit) + split) * D + d] = sum;
    }
    if (tid < G) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += s_red[kWarps * G * D + w * G + tid];
      a.part_l[prow + int64_t(tid) * a.nsplit + split] = sum;
    }
  }
  T* outp = static_cast<T*>(a.out) + (int64_t(b) * a.H_q + int64_t(h) * G) * D;
  if (a.nsplit == 1) {                                     // one split: normalise and write
    for (int idx = tid; idx < G * D; idx += kThreads) {
      float o = 0.f, l = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        o += s_red[w * G * D + idx];
        l += s_red[kWarps * G * D + w * G + idx / D];
      }
      reinterpret_cast<uint16_t*>(outp)[idx] = E::from_f(l > 0.f ? o / l : 0.f);
    }
    return;
  }
  if constexpr (kCluster) {
    // The unit's splits form one cluster; CTA r adds the slice
    // [r * chunk, (r + 1) * chunk) of the G*D outputs. Each CTA stores its
    // partial of every slice (sum p v), and its sum p of every row, into the
    // owner's receive area (past the entries; nothing else uses it, so a peer
    // may store there while this CTA still runs its tokens); one barrier phase
    // (release / acquire) makes the stores visible and each owner adds the
    // partials in split order from its own shared memory.
    const int ns = a.nsplit, n_el = G * D, chunk = (n_el + ns - 1) / ns;
    const uint32_t me = cluster_rank();
    float* rv_o = reinterpret_cast<float*>(s_ent + a.ent_cap);   // [ns][chunk]
    float* rv_l = rv_o + n_el + kMaxClusterSplits;                // [ns][16]
    const uint32_t o_base = smem_u32(rv_o), l_base = smem_u32(rv_l);
    cluster_wait();                                        // every peer has started (the arrive at entry)
    for (int idx = tid; idx < n_el; idx += kThreads) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) o += s_red[w * G * D + idx];
      const int dst = idx / chunk;
      dsmem_st_f32(dsmem_map(o_base + 4u * (me * uint32_t(chunk) + uint32_t(idx - dst * chunk)), uint32_t(dst)), o);
    }
    for (int i = tid; i < ns * G; i += kThreads) {
      const int dst = i / G, g = i - dst * G;
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) l += s_red[kWarps * G * D + w * G + g];
      dsmem_st_f32(dsmem_map(l_base + 4u * (me * 16u + uint32_t(g)), uint32_t(dst)), l);
    }
    cluster_sync();
    const int e0 = int(me) * chunk, e1 = min(n_el, e0 + chunk);
    for (int idx = e0 + tid; idx < e1; idx += kThreads) {
      const int off = idx - e0, row = idx / D;
      float ov[kMaxClusterSplits], lv[kMaxClusterSplits];
#pragma unroll
      for (int r = 0; r < kMaxClusterSplits; ++r) {
        ov[r] = r < ns ? rv_o[r * chunk + off] : 0.f;
        lv[r] = r < ns ? rv_l[r * 16 + row] : 0.f;
      }
      float o = 0.f, l = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxClusterSplits; ++r) { o += ov[r]; l += lv[r]; }   // split order
      reinterpret_cast<uint16_t*>(outp)[idx] = E::from_f(l > 0.f ? o / l : 0.f);
    }
    return;
  }
  // the last split of this (request, KV head) adds the partials in split order
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int done = atomicAdd(&a.tickets[b * a.H_u + h], 1);
    s_last = done == a.nsplit - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < G) {
    float l = 0.f;
#pragma unroll 8
    for (int s = 0; s < a.nsplit; ++s) l += __ldcg(&a.part_l[prow + int64_t(tid) * a.nsplit + s]);
    s_l[tid] = l;
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, d = idx % D;
    const float* src = a.part_o + (prow + int64_t(g) * a.nsplit) * D + d;
    float o = 0.f;
#pragma unroll 8
    for (int s = 0; s < a.nsplit; ++s) o += __ldcg(src + int64_t(s) * D);
    const float l = s_l[g];
    const float y = l > 0.f ? o / l : 0.f;                 // no kept token: 0
    reinterpret_cast<uint16_t*>(outp)[g * D + d] = E::from_f(y);
  }
  if (tid == 0) a.tickets[b * a.H_u + h] = 0;             // ready for the next call
}

struct EntLayout {
  int nsplit, ent_cap;
  size_t logits, tau, part_o, part_l, tickets, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// splits: as many as fit two CTAs per SM in one wave over all (request, KV
// head) units, at least 128 tokens a split, at most one cluster's worth
EntLayout ent_layout(int B, int H_kv, int H_q, int D, int ps, int sel_stride, int sms) {
  EntLayout w;
  const int64_t rows = int64_t(sel_stride) * ps;
  const int units = B * H_kv;
  int ns = (2 * sms) / units;
  const int64_t by_len = (rows + 127) / 128;
  if (ns > by_len) ns = int(by_len);
  if (ns > kMaxClusterSplits) ns = kMaxClusterSplits;
  if (ns < 1) ns = 1;
  w.nsplit = ns;
  const int64_t per = (((rows + ns - 1) / ns) + 31) & ~int64_t(31);
  w.ent_cap = int(per / ps + 2);
  size_t off = 0;
  w.logits = off;  off = align256(off + size_t(B) * H_q * rows * sizeof(float));
  w.tau = off;     off = align256(off + size_t(B) * H_q * sizeof(float));
  w.part_o = off;  off = align256(off + size_t(B) * H_q * ns * D * sizeof(float));
  w.part_l = off;  off = align256(off + size_t(B) * H_q * ns * sizeof(float));
  w.tickets = off; off = align256(off + size_t(B) * H_kv * sizeof(int32_t));
  w.total = off;
  return w;
}

int g_att_smem[16][128];                  // [variant][device] ticket kernels, [variant][64 + device] cluster

template <typename T, int D, int kG>
sa_status launch_attend(const EntArgs& a, dim3 grid, cudaStream_t s, int* attr) {
  const int64_t smem64 = attend_smem(a.G, D, a.ent_cap);
  if (smem64 > 227 * 1024) return SA_ERR_UNSUPPORTED;
  const int smem = int(smem64);
  if (a.nsplit > 1) {                                      // the cluster merge where it can launch
    auto kc = entmax_attend_kernel<T, D, kG, true>;
    if (ensure_smem(kc, smem, attr + 64) &&
        launch_ex(kc, grid, dim3(kThreads), size_t(smem), s, true, unsigned(a.nsplit), a) == cudaSuccess)
      return SA_OK;
    (void)cudaGetLastError();                              // refused: the ticket merge
  }
  auto kt = entmax_attend_kernel<T, D, kG, false>;
  if (!ensure_smem(kt, smem, attr)) return SA_ERR_CUDA;
  return launch_ex(kt, grid, dim3(kThreads), size_t(smem), s, true, 1u, a) == cudaSuccess ? SA_OK
                                                                                      : SA_ERR_CUDA;
}

template <typename T, int D>
sa_status launch_attend_g(const EntArgs& a, dim3 grid, cudaStream_t s, int slot) {
  if (a.G == 1) return launch_attend<T, D, 1>(a, grid, s, g_att_smem[slot * 4 + 3]);
  if (a.G <= 4) return launch_attend<T, D, 4>(a, grid, s, g_att_smem[slot * 4 + 0]);
  if (a.G <= 8) return launch_attend<T, D, 8>(a, grid, s, g_att_smem[slot * 4 + 1]);
  return launch_attend<T, D, 16>(a, grid, s, g_att_smem[slot * 4 + 2]);
}

}  // namespace
}  // namespace sa

extern "C" size_t sa_entmax_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t num_q_heads,
                                           int32_t head_dim, int32_t page_size, int32_t sel_stride) {
  using namespace sa;
  if (batch <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      sel_stride <= 0 || num_q_heads % num_kv_heads)
    return 0;
  return ent_layout(batch, num_kv_heads, num_q_heads, head_dim, page_size, sel_stride, sm_count())
      .total;
}

namespace sa {
namespace {

// per_query_head: the selection has one row per query head (sel [B, H_q,
// stride]); each query head is a unit of one head attending its own pages
// of KV head g / G.
sa_status entmax_impl(const sa_cache* cache, const sa_batch* batch, const void* q, int32_t num_q_heads,
                      const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_stride, float alpha,
                      float scale, void* out, float* tau, float* logits, int32_t logits_stride,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream,
                      bool per_query_head) {
  sa_status st = check_cache(cache, true, false);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (!q || !sel_idx || !sel_cnt || !out || sel_stride <= 0) return SA_ERR_INVALID_ARG;
  if (!aligned16(q)) return SA_ERR_INVALID_ARG;
  if (!(alpha > 1.0f && alpha <= 2.0f)) return SA_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return SA_ERR_INVALID_ARG;
  const int G_kv = num_q_heads / cache->num_kv_heads;
  if (G_kv > 16) return SA_ERR_UNSUPPORTED;
  const int G = per_query_head ? 1 : G_kv;
  const int H_u = per_query_head ? num_q_heads : cache->num_kv_heads;
  const int64_t rows = int64_t(sel_stride) * cache->page_size;
  if (rows > (int64_t(1) << 24)) return SA_ERR_UNSUPPORTED;
  if (logits && logits_stride < rows) return SA_ERR_INVALID_ARG;
  const EntLayout w = ent_layout(batch->batch, H_u, num_q_heads, cache->head_dim, cache->page_size,
                                 sel_stride, sm_count());
  if (!workspace || workspace_bytes < w.total) return SA_ERR_WORKSPACE;
  if (attend_smem(G, cache->head_dim, w.ent_cap) > 227 * 1024) return SA_ERR_UNSUPPORTED;   // (checked before any launch)
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* lg = logits ? logits : reinterpret_cast<float*>(ws + w.logits);
  const int lg_stride = logits ? logits_stride : int(rows);
  // the split counters start at zero (a zero-filled workspace); each call's
  // last CTA per unit leaves its counter at zero again
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // (1) the logits of every selected token (K only)
  st = decode_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, sel_stride, scale, out, nullptr, lg,
                   lg_stride, nullptr, 0, dev_status, stream, /*allow_cluster=*/false, /*pdl=*/false,
                   per_query_head, /*logits_only=*/true);
  if (st != SA_OK) return st;
  EntArgs a;
  a.v = cache->v; a.bt = batch->block_table; a.seq_lens = batch->seq_lens; a.sel = sel_idx;
  a.cnt = sel_cnt; a.logits = lg; a.tau = reinterpret_cast<float*>(ws + w.tau); a.tau_out = tau;
  a.part_o = reinterpret_cast<float*>(ws + w.part_o); a.part_l = reinterpret_cast<float*>(ws + w.part_l);
  a.tickets = reinterpret_cast<int32_t*>(ws + w.tickets);
  a.out = out; a.status = dev_status;
  a.H_kv = cache->num_kv_heads; a.H_q = num_q_heads; a.G = G; a.ps = cache->page_size;
  a.ps_shift = log2i(cache->page_size); a.num_blocks = cache->num_blocks;
  a.bt_stride = batch->bt_stride; a.sel_stride = sel_stride; a.logits_stride = lg_stride;
  a.nsplit = w.nsplit; a.ent_cap = w.ent_cap; a.alpha = alpha;
  a.H_u = H_u; a.kv_div = per_query_head ? G_kv : 1;
  // (2) tau per (request, query head)
  if (launch_ex(entmax_tau_kernel, dim3(unsigned(num_q_heads), unsigned(batch->batch)), dim3(kThreads),
                0, s, true, 1u, a) != cudaSuccess)
    return SA_ERR_CUDA;
  // (3) the kept tokens' sum_j p_j v_j per split, the last split normalising
  const dim3 grid(unsigned(w.nsplit), unsigned(H_u), unsigned(batch->batch));
  const bool bf = cache->dtype == SA_BF16;
  if (cache->head_dim == 128)
    return bf ? launch_attend_g<__nv_bfloat16, 128>(a, grid, s, 0) : launch_attend_g<__half, 128>(a, grid, s, 1);
  return bf ? launch_attend_g<__nv_bfloat16, 64>(a, grid, s, 2) : launch_attend_g<__half, 64>(a, grid, s, 3);
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_sparse_decode_entmax(const sa_cache* cache, const sa_batch* batch,
                                             const void* q, int32_t num_q_heads,
                                             const int32_t* sel_idx, const int32_t* sel_cnt,
                                             int32_t sel_stride, float alpha, float scale, void* out,
                                             float* tau, float* logits, int32_t logits_stride,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, void* stream) {
  return sa::entmax_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, sel_stride, alpha, scale, out,
                         tau, logits, logits_stride, workspace, workspace_bytes, dev_status, stream, false);
}

extern "C" sa_status sa_sparse_decode_entmax_qh(const sa_cache* cache, const sa_batch* batch,
                                                const void* q, int32_t num_q_heads,
                                                const int32_t* sel_idx, const int32_t* sel_cnt,
                                                int32_t sel_stride, float alpha, float scale,
                                                void* out, float* tau, float* logits,
                                                int32_t logits_stride, void* workspace,
                                                size_t workspace_bytes, int32_t* dev_status,
                                                void* stream) {
  return sa::entmax_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, sel_stride, alpha, scale, out,
                         tau, logits, logits_stride, workspace, workspace_bytes, dev_status, stream, true);
}
