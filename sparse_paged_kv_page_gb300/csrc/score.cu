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
// with qbar, P, N the group means of q, q+, q-: 3 FMAs per element whatever
// G is. The kernel is then a gather of 3 * head_dim * 2 bytes of statistics
// per (page, KV head) through the block table, bounded by HBM bandwidth.
//
// Design: persistent CTAs (two per SM). A block's statistics for all KV heads
// are one contiguous run (head after head), so the KV heads are taken Hc at a
// time (Hc = gcd(H_kv, consumer lane groups)) and the pages into chunks of
// 32 / Hc pages x Hc heads: 32 (page, head) pairs per chunk, one TMA copy of
// Hc heads' rows per page. The chunk space runs over the block table's row
// width, page-major (page run, then request, then head group): CTAs working
// at the same time read the same logical pages of every request, whose blocks
// a serving loop that appends to all requests together allocates near each
// other, so the gathers keep some DRAM locality (on the long-context workload
// the scorer takes ~39 us this way against ~43 us request by request). A
// chunk's block ids can be requested before the lengths are known -- the two
// loads overlap at start-up -- and chunks past a request's length are
// skipped. CTA i takes chunks i, i + grid, ... In each CTA one producer warp
// resolves a chunk's block ids and has the TMA engine gather the pages with
// one cp.async.bulk each into a shared-memory ring, completion counted in
// bytes on the stage's mbarrier; four consumer warps score from shared memory
// (D/8 lanes per (page, head), one 16-byte slice of each row per lane,
// shuffle reduction; a lane group always serves the same head of the group,
// so its query coefficients stay in registers) and release the stage. Block
// ids of the next chunk are loaded while the current one is copied; a header
// with a negative count tells the consumers the producer is done.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

#ifndef SA_SCORE_CONSUMER_WARPS
#define SA_SCORE_CONSUMER_WARPS 4
#endif
#ifndef SA_SCORE_STAGES
#define SA_SCORE_STAGES 4
#endif
#ifndef SA_SCORE_CTAS_PER_SM
#define SA_SCORE_CTAS_PER_SM 2
#endif
constexpr int kConsumerWarps = SA_SCORE_CONSUMER_WARPS;
constexpr int kScThreads = 32 * (kConsumerWarps + 1);
constexpr int kChunk = 32;                 // pages per stage (one per producer lane)
constexpr int kStages = SA_SCORE_STAGES;
constexpr int kCtasPerSm = SA_SCORE_CTAS_PER_SM;
constexpr int kMaxBatch = 1024;

struct ScoreArgs {
  const void* meta;
  const void* q;
  const int32_t* bt;
  const int32_t* seq_lens;
  float* scores;
  int32_t* status;
  int B, H_kv, H_q, G, ps, num_blocks, bt_stride, max_pages;
  int hc_shift;                                            // log2(heads per chunk)
  int cpr;                                                 // chunks per (request, head group) row
  float w_avg, w_peak;
};

// kQH: one score per query head (no group mean); its query coefficients for
// G <= 16 heads live in a shared-memory table after a 3-stage ring.
template <int D, bool kQH = false>
struct ScoreTile {
  static constexpr int kPageBytes = 3 * D * 2;             // min, max, mean rows
  // per-query-head pages sit 16 bytes apart beyond their rows so that eight
  // of them read at one column by ldmatrix hit eight different bank groups
  static constexpr int kPageStride = kQH ? kPageBytes + 16 : kPageBytes;
  static constexpr int kStageBytes = kChunk * kPageStride;
  static constexpr int kNStages = kQH ? 3 : kStages;
  static constexpr int kCoefRow = (3 * D + 8) * 2;         // padded coefficient row, bytes
  static constexpr int kCoefBytes = kQH ? 2 * 16 * kCoefRow : 0;
  static constexpr int kSmem = kNStages * kStageBytes + kCoefBytes;
};

struct ChunkHdr {
  int b, hg, p0, count;                                    // request, head group, pages p0 .. +count
  uint32_t valid;                                          // bit j: page p0+j has a good block
};                                                         // count < 0: no more chunks

template <typename T, int D, bool kQH>
__global__ void __maxnreg__(128) score_kernel(ScoreArgs a) {
  using E = Elem<T>;
  using TL = ScoreTile<D, kQH>;
  constexpr int NS = TL::kNStages;
  constexpr int LPP = D / 8;                               // lanes per page
  constexpr int PPP = 32 * kConsumerWarps / LPP;           // pages per consumer pass
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t coef_bar;               // per-head mode: consumers meet here
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ ChunkHdr hdr[kStages];
  __shared__ int s_pages[kMaxBatch];                       // pages of request b (clamped to the row)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hcs = a.hc_shift, Hc = 1 << hcs;
  const int P = kChunk >> hcs;                             // pages per chunk
  const int n_hg = a.H_kv >> hcs;                          // head groups
  const int cap = min(a.max_pages, a.bt_stride);
  const int per_req = n_hg * a.cpr;
  const int total = a.B * per_req;                         // the chunk space
  // chunk c: page run k = c / (B n_hg) (pages kP .. kP+P-1), then request,
  // then head group -- page-major, so CTAs working at the same time read
  // the same logical pages of every request
  auto locate = [&](int c, int& b, int& hg, int& p0) {
    const int k = c / (a.B * n_hg);
    const int r = c - k * (a.B * n_hg);
    b = r / n_hg;
    hg = r - b * n_hg;
    p0 = k * P;
  };
  pdl_wait();

  // The producer's chunks are blockIdx.x, blockIdx.x + gridDim.x, ...; the
  // block ids of its first one are requested before the lengths are known.
  int x_cur = blockIdx.x, cb = 0, cg = 0, cp0 = 0, ck = -1;
  if (warp == kConsumerWarps && x_cur < total) {
    locate(x_cur, cb, cg, cp0);
    ck = (lane < P && cp0 + lane < cap) ? a.bt[int64_t(cb) * a.bt_stride + cp0 + lane] : -1;
  }
  for (int b = tid; b < a.B; b += kScThreads) {
    const int L = a.seq_lens[b];
    const int n_all = L > 0 ? (L + a.ps - 1) / a.ps : 0;
    if (n_all > cap && blockIdx.x == 0) flag(a.status, SA_DEV_OVERFLOW);
    s_pages[b] = min(n_all, cap);
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kConsumerWarps);
    }
    mbar_init(smem_u32(&coef_bar), 32 * kConsumerWarps);
    mbar_init_fence();
  }
  __syncthreads();
  // every length this CTA needs is in shared memory: a programmatically
  // launched successor (the step's append) may start now
  pdl_trigger();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Chunk x_cur is being copied while the block ids of the next one load.
    bool ok = true;
    int it = 0;                                               // stages used (non-empty chunks)
    while (x_cur < total) {
      const int x_nxt = x_cur + int(gridDim.x);
      int nb = 0, ng = 0, np0 = 0, nk = -1;
      if (x_nxt < total) {
        locate(x_nxt, nb, ng, np0);
        nk = (lane < P && np0 + lane < cap) ? a.bt[int64_t(nb) * a.bt_stride + np0 + lane] : -1;
      }
      const int count = min(P, s_pages[cb] - cp0);
      if (count > 0) {
        const int s = it % NS;
        // the stage is free once the consumers released the chunk NS before
        // (one lane waits; the warp takes its answer)
        int freed = 1;
        if (it >= NS && lane == 0) freed = mbar_wait(smem_u32(&empty_bar[s]), ((it / NS) - 1) & 1, a.status);
        if (!__shfl_sync(kFull, freed, 0)) {
          ok = false;
          break;
        }
        const bool good = lane < count && ck >= 0 && ck < a.num_blocks;
        if (lane < count && !good) flag(a.status, SA_DEV_BAD_BLOCK);
        const uint32_t valid = __ballot_sync(kFull, good);
        const uint32_t bytes = uint32_t(TL::kPageBytes) << hcs;   // Hc heads of one block
        if (lane == 0) {
          hdr[s] = ChunkHdr{cb, cg, cp0, count, valid};
          mbar_arrive_expect_tx(smem_u32(&full_bar[s]), uint32_t(__popc(valid)) * bytes);
        }
        __syncwarp();
        if (good) {
          const uint8_t* src = static_cast<const uint8_t*>(a.meta) +
                               (int64_t(ck) * a.H_kv + (cg << hcs)) * int64_t(TL::kPageBytes);
          bulk_g2s(smem_u32(smem + s * TL::kStageBytes + lane * (kQH ? uint32_t(TL::kPageStride) : bytes)),
                   src, bytes, smem_u32(&full_bar[s]));
        }
        ++it;
      }
      x_cur = x_nxt; cb = nb; cg = ng; cp0 = np0; ck = nk;
    }
    // Drain: wait (bounded) until the consumers have released the last
    // stages -- so no copy is in flight -- then tell them there is nothing
    // more (a header with count -1 in the next stage, whose previous chunk is
    // released).
    if (lane == 0) {
      for (int j = max(0, it - NS); j < it && ok; ++j)
        ok = mbar_wait(smem_u32(&empty_bar[j % NS]), (j / NS) & 1, a.status);
      if (ok) {
        const int s = it % NS;
        hdr[s] = ChunkHdr{0, 0, 0, -1, 0u};
        mbar_arrive(smem_u32(&full_bar[s]));
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  if constexpr (kQH) {
    // One score per query head, as a small dense product on the tensor cores:
    // S[g, page] = sum_k A[g, k] B[k, page] with k over the page's 3D
    // statistics (min | max | mean) and A[g] = (w_peak q_g^-, w_peak q_g^+,
    // w_avg q_g). A is held in the element type as two terms, hi = round(A)
    // and lo = round(A - hi) (about 16 significant bits), in rows g and g + 8
    // of a 16-row tile, so one m16n8k16 product accumulates both in float32
    // and their sum is the score. The table is rebuilt whenever the chunk's
    // (request, KV head) changes, the consumers meeting on a bounded mbarrier
    // around the rebuild. Warp w takes pages 8w .. 8w+7 of the chunk (Hc = 1,
    // 32 pages).
    constexpr int KD = 3 * D;
    uint8_t* coef = smem + NS * TL::kStageBytes;          // [mtile][16 rows][KD + 8] elements
    const uint32_t coef_s = smem_u32(coef);
    const int mtiles = a.G > 8 ? 2 : 1;
    const uint32_t cb = smem_u32(&coef_bar);
    uint32_t cphase = 0;
    bool alive = true;
    auto meet = [&]() {
      mbar_arrive(cb);
      alive = alive && mbar_wait(cb, cphase, a.status);
      cphase ^= 1u;
    };
    int cur_b = -1, cur_h = -1;
    const int g4 = lane >> 2, t4 = lane & 3;
    for (int it = 0; alive; ++it) {
      const int s = it % NS;
      if (!__all_sync(kFull, mbar_wait(smem_u32(&full_bar[s]), (it / NS) & 1, a.status))) break;
      const ChunkHdr hd = hdr[s];
      if (hd.count < 0) break;                   // the producer has no more chunks
      const int head = hd.hg;
      if (hd.b != cur_b || head != cur_h) {
        if (cur_b >= 0) meet();                  // every consumer is done with the old table
        cur_b = hd.b;
        cur_h = head;
        const uint16_t* qh = static_cast<const uint16_t*>(a.q) + (int64_t(cur_b) * a.H_q + int64_t(cur_h) * a.G) * D;
        for (int idx = tid; idx < mtiles * 8 * KD; idx += 32 * kConsumerWarps) {
          const int mt = idx / (8 * KD), r = (idx / KD) % 8, k = idx % KD;
          const int g = mt * 8 + r;
          float c = 0.f;
          if (g < a.G) {
            const float x = E::to_f(qh[g * D + (k % D)]);
            c = k < D ? a.w_peak * fminf(x, 0.f) : (k < 2 * D ? a.w_peak * fmaxf(x, 0.f) : a.w_avg * x);
          }
          const uint16_t hi = E::from_f(c);
          const uint16_t lo = E::from_f(c - E::to_f(hi));
          uint16_t* row = reinterpret_cast<uint16_t*>(coef + (mt * 16 + r) * TL::kCoefRow);
          row[k] = hi;
          row[8 * TL::kCoefRow / 2 + k] = lo;    // row r + 8
        }
        meet();                                  // the new table is complete
        if (!alive) break;
      }
      const int j0 = warp * 8;
      if (j0 < hd.count) {
        const uint32_t st = smem_u32(smem + s * TL::kStageBytes);
        // B rows: pages j0 .. j0+7 (lanes 0-7: k 0-7 of the step, lanes 8-15: k 8-15)
        const uint32_t baddr = st + (j0 + (lane & 7)) * TL::kPageStride + ((lane >> 3) & 1) * 16;
        // A rows: lane L addresses row (L>>3 & 1) * 8 + (L & 7), k offset (L >> 4) * 8
        const uint32_t aaddr = coef_s + (((lane >> 3) & 1) * 8 + (lane & 7)) * TL::kCoefRow + (lane >> 4) * 16;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 4
        for (int kk = 0; kk < KD / 16; ++kk) {
          uint32_t bfr[2];
          asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                       : "=r"(bfr[0]), "=r"(bfr[1])
                       : "r"(baddr + kk * 32));
          uint32_t afr[4];
          ldmatrix_x4(afr, aaddr + kk * 32);
          E::mma(acc[0], afr, bfr[0], bfr[1]);
          if (mtiles > 1) {
            ldmatrix_x4(afr, aaddr + 16 * TL::kCoefRow + kk * 32);
            E::mma(acc[1], afr, bfr[0], bfr[1]);
          }
        }
        // this lane: query heads mt*8 + g4, pages j0 + 2*t4 and j0 + 2*t4 + 1
        for (int mt = 0; mt < mtiles; ++mt) {
          const int g = mt * 8 + g4;
          if (g >= a.G) continue;
          float* out = a.scores + (int64_t(hd.b) * a.H_q + int64_t(head) * a.G + g) * a.max_pages + hd.p0;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = j0 + 2 * t4 + e;
            if (j < hd.count)
              out[j] = ((hd.valid >> j) & 1u) ? acc[mt][e] + acc[mt][2 + e] : __int_as_float(0x7fc00000);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
    }
    return;
  }

  // lane group grp serves (page, head) pairs grp, grp + PPP, ... of a chunk;
  // PPP is a multiple of Hc, so its head within the group is always grp % Hc
  const int grp = tid / LPP, l = tid % LPP;
  const int hl = grp & (Hc - 1);
  float ca[8], cp[8], cn[8];
  int cur_b = -1, cur_h = -1;
  for (int it = 0;; ++it) {
    const int s = it % NS;
    if (!__all_sync(kFull, mbar_wait(smem_u32(&full_bar[s]), (it / NS) & 1, a.status))) break;
    const ChunkHdr hd = hdr[s];
    if (hd.count < 0) break;                     // the producer has no more chunks
    const int head = (hd.hg << hcs) + hl;
    if (hd.b != cur_b || head != cur_h) {
      cur_b = hd.b;
      cur_h = head;
#pragma unroll
      for (int e = 0; e < 8; ++e) ca[e] = cp[e] = cn[e] = 0.f;
      const T* qh = static_cast<const T*>(a.q) + (int64_t(cur_b) * a.H_q + int64_t(cur_h) * a.G) * D + l * 8;
      uint4 qv[16];
#pragma unroll
      for (int g = 0; g < 16; ++g)
        qv[g] = g < a.G ? *reinterpret_cast<const uint4*>(qh + int64_t(g) * D) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        if (g >= a.G) break;
        const uint4 v = qv[g];
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
    }
    float* out = a.scores + (int64_t(hd.b) * a.H_kv + head) * a.max_pages + hd.p0;
    const uint8_t* st = smem + s * TL::kStageBytes;
#pragma unroll
    for (int pass = 0; pass < kChunk / PPP; ++pass) {
      const int ph = pass * PPP + grp;                     // (page, head) pair of the chunk
      const int j = ph >> hcs;                             // its page
      const bool here = j < hd.count && ((hd.valid >> j) & 1u);
      float acc = 0.f;
      if (here) {
        const uint8_t* pg = st + ph * TL::kPageStride + l * 16;
        const uint4 vmn = *reinterpret_cast<const uint4*>(pg);
        const uint4 vmx = *reinterpret_cast<const uint4*>(pg + D * 2);
        const uint4 vme = *reinterpret_cast<const uint4*>(pg + 2 * D * 2);
        const uint32_t m0[4] = {vmn.x, vmn.y, vmn.z, vmn.w};
        const uint32_t m1[4] = {vmx.x, vmx.y, vmx.z, vmx.w};
        const uint32_t m2[4] = {vme.x, vme.y, vme.z, vme.w};
        float acc_p = 0.f, acc_n = 0.f;                    // three independent FMA chains
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(ca[2 * e], E::lo(m2[e]), acc);
          acc = fmaf(ca[2 * e + 1], E::hi(m2[e]), acc);
          acc_p = fmaf(cp[2 * e], E::lo(m1[e]), acc_p);
          acc_p = fmaf(cp[2 * e + 1], E::hi(m1[e]), acc_p);
          acc_n = fmaf(cn[2 * e], E::lo(m0[e]), acc_n);
          acc_n = fmaf(cn[2 * e + 1], E::hi(m0[e]), acc_n);
        }
        acc += acc_p + acc_n;
      }
#pragma unroll
      for (int o = LPP / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      if (l == 0 && j < hd.count) out[j] = here ? acc : __int_as_float(0x7fc00000);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
  }
}

// ---------------------------------------------------------------------------
// Per-query-head scores for G <= 8 without a shared-memory ring
// ---------------------------------------------------------------------------
#ifndef SA_QH_GROUPS
#define SA_QH_GROUPS 16
#endif
constexpr int kQhWarps = 4;
constexpr int kQhGroups = SA_QH_GROUPS;                    // 8-page groups per warp

// The same product S[g, page] = sum_k A[g, k] B[k, page] over the page's 3D
// statistics, one warp per run of kQhGroups groups of 8 pages of one
// (request, KV head), the pages the n columns of m16n8k16. The sum over k may
// take the statistics in any order, so lane (g4, t4) reads, of page g4 of the
// group, the 16-byte pieces at byte offsets 64 i + 16 t4 of its 3D-element
// row (the four lanes of a page read 64 contiguous bytes per load) straight
// into B fragments: piece i fills k steps 2 i (its first 4 elements) and
// 2 i + 1 (the next 4). A, built once per warp in that order, holds head g4's
// coefficient hi in row g4 and lo in row g4 + 8, so the score of head g4 at
// page j is the sum of the two rows. The next group's rows are loaded while
// the current one is multiplied.
template <typename T, int D>
__global__ void __launch_bounds__(32 * kQhWarps, 2) score_qh_kernel(ScoreArgs a) {
  using E = Elem<T>;
  constexpr int KD = 3 * D;
  constexpr int NP = KD / 32;                              // pieces per lane per row
  constexpr int KS = KD / 16;                              // k steps
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g4 = lane >> 2, t4 = lane & 3;
  pdl_wait();
  const int L = a.seq_lens[b];
  pdl_trigger();
  const int n_all = L > 0 ? (L + a.ps - 1) / a.ps : 0;
  const int cap = min(a.max_pages, a.bt_stride);
  if (n_all > cap && blockIdx.x == 0 && h == 0 && threadIdx.x == 0) flag(a.status, SA_DEV_OVERFLOW);
  const int n = min(n_all, cap);
  const int base = (blockIdx.x * kQhWarps + warp) * (8 * kQhGroups);
  if (base >= n) return;

  int blk[kQhGroups];
#pragma unroll
  for (int gi = 0; gi < kQhGroups; ++gi) {
    const int p = base + 8 * gi + g4;
    blk[gi] = p < n ? a.bt[int64_t(b) * a.bt_stride + p] : -1;
  }
  // A fragments: k step 2 i + hf covers elements 32 i + 8 t4 + 4 hf + {0, 1} (a0 / a1)
  // and + {2, 3} (a2 / a3) of the coefficient row (w_peak q- | w_peak q+ | w_avg q)
  uint32_t af[KS][4];
  {
    const uint16_t* qh = static_cast<const uint16_t*>(a.q) + (int64_t(b) * a.H_q + int64_t(h) * a.G + g4) * D;
    const bool live = g4 < a.G;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int k0 = 32 * i + 8 * t4;                      // first element of this lane's piece
      const int third = k0 / D, d0 = k0 % D;
      const uint4 u = live ? *reinterpret_cast<const uint4*>(qh + d0) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float c[2];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
          const float x = z ? E::hi(w[e]) : E::lo(w[e]);
          c[z] = third == 0 ? a.w_peak * fminf(x, 0.f) : (third == 1 ? a.w_peak * fmaxf(x, 0.f) : a.w_avg * x);
        }
        const uint32_t hv = E::pack(c[0], c[1]);
        hi[e] = hv;
        lo[e] = E::pack(c[0] - E::lo(hv), c[1] - E::hi(hv));
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        af[2 * i + hf][0] = hi[2 * hf];
        af[2 * i + hf][1] = lo[2 * hf];
        af[2 * i + hf][2] = hi[2 * hf + 1];
        af[2 * i + hf][3] = lo[2 * hf + 1];
      }
    }
  }
  const uint4* meta4 = static_cast<const uint4*>(a.meta);
  auto good = [&](int bk) { return bk >= 0 && bk < a.num_blocks; };
  auto load = [&](int bk, uint4 (&r)[NP]) {
    const int64_t row = (int64_t(bk) * a.H_kv + h) * (KD / 8);
#pragma unroll
    for (int i = 0; i < NP; ++i) r[i] = good(bk) ? __ldg(meta4 + row + 4 * i + t4) : make_uint4(0u, 0u, 0u, 0u);
  };
  uint4 cur[NP];
  load(blk[0], cur);
#pragma unroll
  for (int gi = 0; gi < kQhGroups; ++gi) {
    const int p0 = base + 8 * gi;
    if (p0 >= n) break;
    uint4 nxt[NP];
    if (gi + 1 < kQhGroups) load(blk[gi + 1], nxt);       // the next group's rows in flight
    if (p0 + g4 < n && !good(blk[gi]) && t4 == 0) flag(a.status, SA_DEV_BAD_BLOCK);
    const uint32_t ok = __ballot_sync(kFull, good(blk[gi]));
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      E::mma(acc, af[2 * i], cur[i].x, cur[i].y);
      E::mma(acc, af[2 * i + 1], cur[i].z, cur[i].w);
    }
    if (g4 < a.G) {
      float* out = a.scores + (int64_t(b) * a.H_q + int64_t(h) * a.G + g4) * a.max_pages + p0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 2 * t4 + e;
        if (p0 + j < n) out[j] = ((ok >> (4 * j)) & 1u) ? acc[e] + acc[2 + e] : __int_as_float(0x7fc00000);
      }
    }
    if (gi + 1 < kQhGroups) {
#pragma unroll
      for (int i = 0; i < NP; ++i) cur[i] = nxt[i];
    }
  }
}

template <typename T, int D>
sa_status launch_score_qh(const ScoreArgs& a, cudaStream_t s) {
  const int per_cta = 8 * kQhGroups * kQhWarps;
  const int cap = a.max_pages < a.bt_stride ? a.max_pages : a.bt_stride;
  const dim3 grid(unsigned((cap + per_cta - 1) / per_cta), unsigned(a.H_kv), unsigned(a.B));
  score_qh_kernel<T, D><<<grid, 32 * kQhWarps, 0, s>>>(a);
  return launch_status();
}

int g_sc_smem[8][64];

template <typename T, int D, bool kQH>
sa_status launch_score(const ScoreArgs& a, int grid, cudaStream_t s, int* cache) {
  auto k = score_kernel<T, D, kQH>;
  if (!ensure_smem(k, ScoreTile<D, kQH>::kSmem, cache)) return SA_ERR_CUDA;
  k<<<grid, kScThreads, ScoreTile<D, kQH>::kSmem, s>>>(a);
  return launch_status();
}

}  // namespace
}  // namespace sa

sa_status sa::score_impl(const sa_cache* cache, const sa_batch* batch, const void* q,
                        int32_t num_q_heads, float w_avg, float w_peak, float* scores,
                        int32_t max_pages, int32_t* dev_status, void* stream, bool per_query_head) {
  using namespace sa;
  sa_status st = check_cache(cache, false, true);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (!q || !scores || max_pages <= 0) return SA_ERR_INVALID_ARG;
  if (!aligned16(q)) return SA_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return SA_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  if (G > 16) return SA_ERR_UNSUPPORTED;
  if (batch->batch > kMaxBatch) return SA_ERR_UNSUPPORTED;
  ScoreArgs a;
  a.meta = cache->meta; a.q = q; a.bt = batch->block_table; a.seq_lens = batch->seq_lens;
  a.scores = scores; a.status = dev_status;
  a.B = batch->batch; a.H_kv = cache->num_kv_heads; a.H_q = num_q_heads; a.G = G;
  a.ps = cache->page_size; a.num_blocks = cache->num_blocks; a.bt_stride = batch->bt_stride;
  a.max_pages = max_pages; a.w_avg = w_avg; a.w_peak = w_peak;
  // heads per chunk: the largest power of two dividing both H_kv and the
  // consumers' lane groups (128 / (head_dim / 8))
  const int groups = 32 * kConsumerWarps / (cache->head_dim / 8);
  int hc = 1;
  while (!per_query_head && hc < groups && a.H_kv % (2 * hc) == 0) hc *= 2;
  a.hc_shift = log2i(hc);
  // the chunk space over the table rows; enough persistent CTAs for two per
  // SM, never more than chunks exist
  const int cap = max_pages < batch->bt_stride ? max_pages : batch->bt_stride;
  const int per_chunk = kChunk / hc;
  a.cpr = (cap + per_chunk - 1) / per_chunk;
  const int64_t max_chunks = int64_t(batch->batch) * (a.H_kv / hc) * a.cpr;
  if (max_chunks > 0x7fffffff - 4 * 1024 * 1024) return SA_ERR_UNSUPPORTED;
  const int full = kCtasPerSm * sm_count();
  const int grid = int(max_chunks < full ? max_chunks : full);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = cache->dtype == SA_BF16;
  if (per_query_head && G <= 8) {
    if (cache->head_dim == 128)
      return bf ? launch_score_qh<__nv_bfloat16, 128>(a, s) : launch_score_qh<__half, 128>(a, s);
    return bf ? launch_score_qh<__nv_bfloat16, 64>(a, s) : launch_score_qh<__half, 64>(a, s);
  }
  if (per_query_head) {
    if (cache->head_dim == 128)
      return bf ? launch_score<__nv_bfloat16, 128, true>(a, grid, s, g_sc_smem[4])
                : launch_score<__half, 128, true>(a, grid, s, g_sc_smem[5]);
    return bf ? launch_score<__nv_bfloat16, 64, true>(a, grid, s, g_sc_smem[6])
              : launch_score<__half, 64, true>(a, grid, s, g_sc_smem[7]);
  }
  if (cache->head_dim == 128)
    return bf ? launch_score<__nv_bfloat16, 128, false>(a, grid, s, g_sc_smem[0])
              : launch_score<__half, 128, false>(a, grid, s, g_sc_smem[1]);
  return bf ? launch_score<__nv_bfloat16, 64, false>(a, grid, s, g_sc_smem[2])
            : launch_score<__half, 64, false>(a, grid, s, g_sc_smem[3]);
}

extern "C" sa_status sa_score_pages(const sa_cache* cache, const sa_batch* batch, const void* q,
                                    int32_t num_q_heads, float w_avg, float w_peak, float* scores,
                                    int32_t max_pages, int32_t* dev_status, void* stream) {
  return sa::score_impl(cache, batch, q, num_q_heads, w_avg, w_peak, scores, max_pages, dev_status,
                        stream, false);
}

extern "C" sa_status sa_score_pages_qh(const sa_cache* cache, const sa_batch* batch, const void* q,
                                       int32_t num_q_heads, float w_avg, float w_peak,
                                       float* scores, int32_t max_pages, int32_t* dev_status,
                                       void* stream) {
  return sa::score_impl(cache, batch, q, num_q_heads, w_avg, w_peak, scores, max_pages, dev_status,
                        stream, true);
}
