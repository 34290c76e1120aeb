// sa_sparse_decode: exact softmax attention over the selected pages only,
// split across CTAs, partials merged by their log-sum-exp.
//
// "EntmaxKV" README, "How it works": only the selected pages are attended and
// the attention is exact over that selection. "flow: add H2O sparse
// attention" (vortex_torch PR 6), "Token-level variants" point 1: softmax
// scale head_dim ** -0.5 unless given. "test_ops_mla_chunked_context.cpp"
// (vllm.cpp): chunked attention merged by log-sum-exp must equal single-shot
// attention; an empty chunk carries lse = -inf.
//
// Work unit: a tile of 16 token rows of one (request, KV head) taken in
// selection order (row i = entry i / page_size, slot i % page_size), so a
// 16-token page is one tile and page_size 1 gathers 16 retained tokens.
// Grid (nsplit, units, B) -- a unit is a KV head with its G query heads, or
// one query head under per-query-head selection: CTA `split` of a unit takes an equal share of the
// unit's tiles, counted on the device from sel_cnt, and first resolves the
// selection entries it touches to (block, fill) in shared memory. Its 4 warps
// take tiles round robin, each with a private ring of stages:
//  * page_size >= 16: a tile is 16 contiguous rows of one (block, head), so
//    the TMA engine fetches it through a 2-D tensor map over all pool rows
//    (cp.async.bulk.tensor, 64-column boxes, 128-byte swizzle), completion
//    on the stage's mbarrier; slots past a page's fill are masked, and the
//    stale V rows of a partial page are zeroed in shared memory;
//  * page_size < 16: rows come from different pages, gathered with 16-byte
//    cp.async (zero-fill for invalid rows) into the same swizzled layout.
// Per tile a warp computes S = Q K^T with mma.sync m16n8k16 (rows = the G
// query heads, padded to 16; columns = the 16 tokens), applies scale and mask,
// runs the online softmax in float32 (exp2 domain), reuses P's accumulator
// registers as the A operand of O += P V, and at the end the 4 warps merge in
// shared memory. Each CTA writes its partial (o_s, lse_s) to the workspace; the
// last CTA of the unit to finish (atomic ticket) merges the partials exactly,
// writes out / lse and resets the ticket. No CTA waits on another; every
// mbarrier wait is time-bounded.
#include <cuda.h>

#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

#ifndef SA_DECODE_STAGES
#define SA_DECODE_STAGES 3
#endif
#ifndef SA_DECODE_CTAS_PER_SM
#define SA_DECODE_CTAS_PER_SM 2
#endif
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = SA_DECODE_STAGES;
constexpr int kCtasPerSm = SA_DECODE_CTAS_PER_SM;
constexpr int kMaxSplit = 64;
constexpr int kMaxCluster = 8;         // portable cluster size: splits merged through DSMEM
constexpr int kMaxEnt = 4096;          // (block, fill) entries staged per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeArgs {
  const void* k;
  const void* v;
  const void* q;
  const int32_t* bt;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* cnt;
  void* out;
  float* lse;
  float* logits;
  float* part_o;
  float* part_lse;
  int32_t* tickets;
  int32_t* status;
  int H_kv, H_q, G, ps, ps_shift, num_blocks, bt_stride, sel_stride, logits_stride, nsplit;
  int H_u, kv_div;  // selection units per request (H_kv, or H_q per query head) and per KV head
  int logits_only;  // write the scaled logits and stop: V is neither read nor used
  int ent_max;      // entries of the selection one CTA can touch
  float scale, scale_log2;
};

// Cluster merge receive area, past the selection entries: every peer's partial
// of the slice this CTA merges ([nsplit][chunk] floats, nsplit * chunk <=
// 16 * D + kMaxCluster) and every peer's lse of each row ([kMaxCluster][16]).
template <int D>
constexpr int recv_bytes() { return 4 * (16 * D + kMaxCluster + kMaxCluster * 16); }
__host__ __device__ constexpr int recv_off(int tile_smem, int ent_max) {
  return (tile_smem + ent_max * 8 + 15) & ~15;
}

// Shared-memory tile of 16 rows x D columns (2-byte elements): 64-column
// halves of 16 x 128 bytes, each 16-byte chunk c of row r stored at chunk
// position c ^ (r & 7) -- the TMA 128-byte swizzle, so 8 rows read at one
// column hit 8 different bank groups.
template <int D>
struct Tile {
  static constexpr int kHalves = D / 64;
  static constexpr int kBytes = 16 * D * 2;          // one K (or V) tile
  static constexpr int kChunks = D / 8;              // 16-byte chunks per row
  static constexpr int kRowsPerOp = 32 / kChunks;    // rows one warp-wide cp.async covers
  static constexpr int kOps = 16 / kRowsPerOp;       // cp.async per lane per tile
  static constexpr int kStageBytes = 2 * kBytes;     // K + V
  static constexpr int kStageArea = kWarps * kStages * kStageBytes;
  // the stage area is reused for the warp-merge scratch: row maxima and sums
  // ([kWarps][16] each) and partial outputs ([kWarps][16][D + 4] floats)
  static constexpr int kMergeArea = 4 * (kWarps * 32 + kWarps * 16 * (D + 4));
  static constexpr int kSmem = (kStageArea > kMergeArea ? kStageArea : kMergeArea) + 1024;   // + alignment slack
};


template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return uint32_t((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <typename T, int D, bool kTma, bool kCluster>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  using E = Elem<T>;
  using TL = Tile<D>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ uint32_t s_mask[kWarps][kStages];
  __shared__ __align__(8) uint64_t s_bar[kWarps][kStages];
  __shared__ int s_last;
  __shared__ float s_sf[kWarps][16];           // per-warp weights of each output row
  __shared__ float s_rl[16];                   // this CTA's lse of each row
  // 1024-byte aligned base for the swizzled tiles
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  // Cluster merge: peers store into this CTA's receive area only after this
  // arrive has been waited on, i.e. once every CTA of the cluster has started.
  const bool push = kCluster && !a.logits_only && a.nsplit > 1;
  if (push) cluster_arrive_relaxed();

  // h: the selection unit within the request -- a KV head with its G query
  // heads, or (per-query-head selection, G = 1) one query head of KV head kvh
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = b * a.H_u + h;
  const int kvh = h / a.kv_div;
  const int G = a.G, ps = a.ps, pss = a.ps_shift;

  // Q as the A operand (rows = query heads of this KV head, zero beyond G).
  // Q is an input of the step, so it is read before waiting on the selection.
  const int g = lane >> 2, tq = lane & 3;
  uint32_t qa[D / 16][4];
  {
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(a.q) + (int64_t(b) * a.H_q + int64_t(h) * G) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c0 = (kk * 16 + 2 * tq) >> 1, c1 = c0 + 4;
      qa[kk][0] = g < G ? qp[g * (D / 2) + c0] : 0u;
      qa[kk][1] = g + 8 < G ? qp[(g + 8) * (D / 2) + c0] : 0u;
      qa[kk][2] = g < G ? qp[g * (D / 2) + c1] : 0u;
      qa[kk][3] = g + 8 < G ? qp[(g + 8) * (D / 2) + c1] : 0u;
    }
  }
  if (kTma && threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&s_bar[w][s]), 1);
    mbar_init_fence();
  }
  // lengths and selection come from the kernels before this one in the step
  pdl_wait();
  if (a.logits_only) pdl_trigger();                           // the entmax threshold kernel may launch

  // This CTA's range of selection entries is a function of the count. The
  // entry it would start at with a full selection (the usual case) is loaded
  // together with the count, so the block lookups start one round trip early;
  // the value is used only if the real range starts there too.
  const int32_t* sel = a.sel + int64_t(unit) * a.sel_stride;
  auto entry_range = [&](int count, int& e_begin, int& e_cnt, int& t_begin, int& t_end, int& n_rows) {
    n_rows = count << pss;
    const int n_tiles = (n_rows + 15) >> 4;
    const int per = (n_tiles + a.nsplit - 1) / a.nsplit;
    t_begin = min(n_tiles, split * per);
    t_end = min(n_tiles, t_begin + per);
    const int row_begin = t_begin << 4, row_end = min(t_end << 4, n_rows);
    e_begin = row_begin >> pss;
    e_cnt = row_end > row_begin ? min(((row_end - 1) >> pss) - e_begin + 1, a.ent_max) : 0;
  };
  int eb_s, ec_s, tb_s, te_s, nr_s;
  entry_range(a.sel_stride, eb_s, ec_s, tb_s, te_s, nr_s);
  const int spec_page = threadIdx.x < ec_s ? sel[eb_s + threadIdx.x] : -1;

  const int L = a.seq_lens[b];
  int cnt = a.cnt[unit];
  if (cnt < 0 || cnt > a.sel_stride) {
    if (threadIdx.x == 0 && split == 0) flag(a.status, SA_DEV_BAD_COUNT);
    cnt = cnt < 0 ? 0 : a.sel_stride;
  }
  int e_begin, e_cnt, t_begin, t_end, n_rows;
  entry_range(cnt, e_begin, e_cnt, t_begin, t_end, n_rows);
  const int row_end = min(t_end << 4, n_rows);
  const int n_pages_req = L > 0 ? (L + ps - 1) >> pss : 0;
  const int32_t* btb = a.bt + int64_t(b) * a.bt_stride;

  // Prologue: resolve the selection entries this CTA touches to (block, fill)
  // once, in parallel, so the copy loop never waits on sel -> block table.
  int2* s_ent = reinterpret_cast<int2*>(smem_raw + TL::kSmem);
  for (int i = threadIdx.x; i < e_cnt; i += kThreads) {
    const int e = e_begin + i;
    int blk = -1, fill = 0;
    const int page = (e == eb_s + int(threadIdx.x) && int(threadIdx.x) < ec_s) ? spec_page : sel[e];
    if (page < 0 || page >= n_pages_req || page >= a.bt_stride) {
      flag(a.status, SA_DEV_BAD_BLOCK);
    } else {
      fill = min(ps, L - (page << pss));
      const int x = btb[page];
      if (x < 0 || x >= a.num_blocks) flag(a.status, SA_DEV_BAD_BLOCK);
      else blk = x;
    }
    s_ent[i] = make_int2(blk, fill);
  }
  __syncthreads();

  float o[D / 8][4];
#pragma unroll
  for (int x = 0; x < D / 8; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  uint8_t* wbuf = smem + warp * kStages * TL::kStageBytes;
  const int nt = t_begin + warp < t_end ? (t_end - t_begin - warp + kWarps - 1) / kWarps : 0;

  // Start the copies of this warp's i-th tile into stage st.
  auto issue = [&](int i, int st) {
    const int t = t_begin + warp + i * kWarps;
    const uint32_t sk = smem_u32(wbuf + st * TL::kStageBytes);
    const uint32_t sv = sk + TL::kBytes;
    if constexpr (kTma) {
      // one (block, head) row range: 16 rows starting at slot s0 of entry e
      const int j0 = t << 4;
      const int ei = (j0 >> pss) - e_begin, s0 = j0 & (ps - 1);
      int y = 0, nvalid = 0;
      if (j0 < row_end && ei < e_cnt) {
        const int2 en = s_ent[ei];
        if (en.x >= 0 && s0 < en.y) {
          nvalid = min(16, en.y - s0);
          y = int((int64_t(en.x) * a.H_kv + kvh) * ps + s0);
        }
      }
      const uint32_t vmask = nvalid >= 16 ? 0xffffu : ((1u << nvalid) - 1u);
      if (lane == 0) {
        s_mask[warp][st] = vmask;
        const uint32_t bar = smem_u32(&s_bar[warp][st]);
        fence_proxy_async_smem();
        const int nbuf = a.logits_only ? 1 : 2;
        mbar_arrive_expect_tx(bar, vmask ? uint32_t(nbuf * TL::kBytes) : 0u);
        if (vmask) {
#pragma unroll
          for (int hf = 0; hf < TL::kHalves; ++hf) {
            tma_load_2d(sk + hf * 2048, &tmk, hf * 64, y, bar);
            if (!a.logits_only) tma_load_2d(sv + hf * 2048, &tmv, hf * 64, y, bar);
          }
        }
      }
    } else {
      int64_t off = 0;
      bool valid = false;
      if (lane < 16) {
        const int j = (t << 4) + lane;
        const int ei = (j >> pss) - e_begin, s = j & (ps - 1);
        if (j < row_end && ei < e_cnt) {
          const int2 en = s_ent[ei];
          if (en.x >= 0 && s < en.y) {
            valid = true;
            off = ((int64_t(en.x) * a.H_kv + kvh) * ps + s) * D;
          }
        }
      }
      const uint32_t vmask = __ballot_sync(kFull, valid) & 0xffffu;
      if (lane == 0) s_mask[warp][st] = vmask;
      const T* kbase = static_cast<const T*>(a.k);
      const T* vbase = static_cast<const T*>(a.v);
      const int chunk = lane % TL::kChunks;
#pragma unroll
      for (int r0 = 0; r0 < TL::kOps; ++r0) {
        const int row = lane / TL::kChunks + r0 * TL::kRowsPerOp;
        const int lo = __shfl_sync(kFull, int(uint64_t(off) & 0xffffffffu), row);
        const int hi = __shfl_sync(kFull, int(uint64_t(off) >> 32), row);
        const int64_t ro = int64_t((uint64_t(uint32_t(hi)) << 32) | uint32_t(lo));
        const bool rv = (vmask >> row) & 1u;
        const uint32_t d = swz<D>(row, chunk);
        cp_async_16(sk + d, rv ? static_cast<const void*>(kbase + ro + chunk * 8) : a.k, rv ? 16 : 0);
        if (!a.logits_only)
          cp_async_16(sv + d, rv ? static_cast<const void*>(vbase + ro + chunk * 8) : a.v, rv ? 16 : 0);
      }
    }
  };

  bool alive = true;
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < nt) issue(i, i);
    if constexpr (!kTma) cp_async_commit();
  }
  for (int i = 0; i < nt && alive; ++i) {
    const int nxt = i + kStages - 1;
    __syncwarp();
    if (nxt < nt) issue(nxt, nxt % kStages);
    const int st = i % kStages;
    if constexpr (kTma) {
      if (!mbar_wait(smem_u32(&s_bar[warp][st]), (i / kStages) & 1, a.status)) { alive = false; break; }
    } else {
      cp_async_commit();
      cp_async_wait<kStages - 1>();
    }
    __syncwarp();
    const int t = t_begin + warp + i * kWarps;
    const uint32_t sk = smem_u32(wbuf + st * TL::kStageBytes);
    const uint32_t sv = sk + TL::kBytes;
    const uint32_t vmask = s_mask[warp][st];
    if (vmask == 0) {
      if (a.logits) {                                          // no valid token in the tile
        const int j = (t << 4) + (lane & 15);
        if (j < n_rows)
          for (int gg = lane >> 4; gg < G; gg += 2)
            a.logits[(int64_t(b) * a.H_q + int64_t(h) * G + gg) * a.logits_stride + j] = -INFINITY;
      }
      continue;
    }
    if (kTma && vmask != 0xffffu && !a.logits_only) {
      // a partial page: its stale V rows could hold anything (NaN) -- zero them
      for (int idx = lane; idx < 16 * TL::kChunks; idx += 32) {
        const int row = idx / TL::kChunks, chunk = idx % TL::kChunks;
        if (!((vmask >> row) & 1u))
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(sv + swz<D>(row, chunk)), "r"(0u)
                       : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
    }

    // S = Q K^T   (c[ntile][.]: rows g / g+8, tokens ntile*8 + 2tq + {0,1})
    float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      // even and odd k-steps accumulate separately: two dependency chains of D/32
      float c2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane >> 3, rr = lane & 7;
      const int tok = (mi >> 1) * 8 + rr;
#pragma unroll
      for (int kk = 0; kk < D / 16; kk += 2) {
        uint32_t r[4], r2[4];
        ldmatrix_x4(r, sk + swz<D>(tok, kk * 2 + (mi & 1)));
        ldmatrix_x4(r2, sk + swz<D>(tok, (kk + 1) * 2 + (mi & 1)));
        E::mma(c[0], qa[kk], r[0], r[1]);
        E::mma(c[1], qa[kk], r[2], r[3]);
        E::mma(c2[0], qa[kk + 1], r2[0], r2[1]);
        E::mma(c2[1], qa[kk + 1], r2[2], r2[3]);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) { c[0][x] += c2[0][x]; c[1][x] += c2[1][x]; }
    }
    // scale, mask, logits, online softmax
    float pmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt2 = 0; nt2 < 2; ++nt2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = nt2 * 8 + 2 * tq + e;
        const bool ok = (vmask >> tok) & 1u;
        const int j = (t << 4) + tok;
        if (a.logits && j < n_rows) {
          float* lg = a.logits + (int64_t(b) * a.H_q + int64_t(h) * G) * a.logits_stride + j;
          if (g < G) lg[int64_t(g) * a.logits_stride] = ok ? c[nt2][e] * a.scale : -INFINITY;
          if (g + 8 < G) lg[int64_t(g + 8) * a.logits_stride] = ok ? c[nt2][2 + e] * a.scale : -INFINITY;
        }
        c[nt2][e] = ok ? c[nt2][e] * a.scale_log2 : -INFINITY;
        c[nt2][2 + e] = ok ? c[nt2][2 + e] * a.scale_log2 : -INFINITY;
        pmax[0] = fmaxf(pmax[0], c[nt2][e]);
        pmax[1] = fmaxf(pmax[1], c[nt2][2 + e]);
      }
    }
    if (a.logits_only) continue;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      pmax[r] = fmaxf(pmax[r], __shfl_xor_sync(kFull, pmax[r], 1));
      pmax[r] = fmaxf(pmax[r], __shfl_xor_sync(kFull, pmax[r], 2));
      const float m_new = fmaxf(m_r[r], pmax[r]);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2_approx(m_r[r] - m_use);
      float rs = 0.f;
#pragma unroll
      for (int nt2 = 0; nt2 < 2; ++nt2) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float p = ex2_approx(c[nt2][2 * r + e] - m_use);
          c[nt2][2 * r + e] = p;
          rs += p;
        }
      }
      l_r[r] = l_r[r] * alpha + rs;
      m_r[r] = m_new;
#pragma unroll
      for (int x = 0; x < D / 8; ++x) { o[x][2 * r] *= alpha; o[x][2 * r + 1] *= alpha; }
    }
    // O += P V
    const uint32_t pa[4] = {E::pack(c[0][0], c[0][1]), E::pack(c[0][2], c[0][3]),
                            E::pack(c[1][0], c[1][1]), E::pack(c[1][2], c[1][3])};
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int tok = (mi & 1) * 8 + rr;
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        uint32_t r[4];
        ldmatrix_x4_trans(r, sv + swz<D>(tok, 2 * nd + (mi >> 1)));
        E::mma(o[2 * nd], pa, r[0], r[1]);
        E::mma(o[2 * nd + 1], pa, r[2], r[3]);
      }
    }
  }
  if constexpr (kTma) {
    // never leave with copies in flight (bounded): drain this warp's issued stages
    if (lane == 0 && !alive) {
      for (int i = 0; i < nt; ++i)
        if (!mbar_wait(smem_u32(&s_bar[warp][i % kStages]), (i / kStages) & 1, a.status)) break;
    }
  } else {
    cp_async_wait<0>();
  }
  if (a.logits_only) return;                                   // (uniform across the CTA)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(kFull, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(kFull, l_r[r], 2);
  }
  __syncthreads();

  // merge the 4 warps in shared memory (reusing the tile buffers): each row's
  // weights once, then one weighted sum per output element
  constexpr int WS = D + 4;                                    // padded row: no bank conflicts
  float* wm = reinterpret_cast<float*>(smem);                 // [kWarps][16] row maxima (log2)
  float* wl = wm + kWarps * 16;                                // [kWarps][16] row sums
  float* wo = wl + kWarps * 16;                                // [kWarps][G][WS]
  if (tq == 0) {
    if (g < G) { wm[warp * 16 + g] = m_r[0]; wl[warp * 16 + g] = l_r[0]; }
    if (g + 8 < G) { wm[warp * 16 + g + 8] = m_r[1]; wl[warp * 16 + g + 8] = l_r[1]; }
  }
#pragma unroll
  for (int x = 0; x < D / 8; ++x) {
    const int d = x * 8 + 2 * tq;
    if (g < G) {
      wo[(warp * G + g) * WS + d] = o[x][0];
      wo[(warp * G + g) * WS + d + 1] = o[x][1];
    }
    if (g + 8 < G) {
      wo[(warp * G + g + 8) * WS + d] = o[x][2];
      wo[(warp * G + g + 8) * WS + d + 1] = o[x][3];
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int row = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * 16 + row]);
    float f[kWarps], tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = wm[w * 16 + row];
      f[w] = mw == -INFINITY ? 0.f : ex2_approx(mw - M);      // a warp without tokens weighs 0
      tot = fmaf(wl[w * 16 + row], f[w], tot);
    }
    const float inv = tot > 0.f ? rcp_approx(tot) : 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s_sf[w][row] = f[w] * inv;
    s_rl[row] = tot > 0.f ? (M + lg2_approx(tot)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  // this CTA's normalised output of element (row, d)
  auto merged = [&](int row, int d) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float sf = s_sf[w][row];
      if (sf != 0.f) acc = fmaf(wo[(w * G + row) * WS + d], sf, acc);
    }
    return acc;
  };
  T* outp = static_cast<T*>(a.out) + (int64_t(b) * a.H_q + int64_t(h) * G) * D;
  if (a.nsplit == 1) {
    for (int idx = threadIdx.x; idx < G * D; idx += kThreads)
      reinterpret_cast<uint16_t*>(outp)[idx] = E::from_f(merged(idx / D, idx % D));
    if (a.lse && threadIdx.x < G) a.lse[int64_t(b) * a.H_q + int64_t(h) * G + threadIdx.x] = s_rl[threadIdx.x];
    return;
  }

  if constexpr (kCluster) {
    // The unit's nsplit CTAs form one cluster; CTA r merges the slice
    // [r * chunk, (r + 1) * chunk) of the unit's G*D outputs. Each CTA stores
    // its partial of every slice, and its lse of every row, into the owner's
    // receive area (a region no tile uses, so a peer may store there while
    // this CTA still streams tiles); one barrier phase (release / acquire)
    // makes the stores visible, and each owner merges from its own shared
    // memory, after which no CTA touches another's shared memory again.
    const int ns = a.nsplit;
    const int n_el = G * D, chunk = (n_el + ns - 1) / ns;
    const uint32_t me = cluster_rank();
    float* rv_o = reinterpret_cast<float*>(smem_raw + recv_off(TL::kSmem, a.ent_max));   // [ns][chunk]
    float* rv_l = rv_o + 16 * D + kMaxCluster;                                          // [ns][16]
    const uint32_t o_base = smem_u32(rv_o), l_base = smem_u32(rv_l);
    cluster_wait();                              // every peer has started (the arrive at entry)
    for (int idx = threadIdx.x; idx < n_el; idx += kThreads) {
      const int dst = idx / chunk;
      dsmem_st_f32(dsmem_map(o_base + 4u * (me * uint32_t(chunk) + uint32_t(idx - dst * chunk)), uint32_t(dst)),
                   merged(idx / D, idx % D));
    }
    for (int i = threadIdx.x; i < ns * G; i += kThreads) {
      const int dst = i / G, row = i - dst * G;
      dsmem_st_f32(dsmem_map(l_base + 4u * (me * 16u + uint32_t(row)), uint32_t(dst)), s_rl[row]);
    }
    cluster_sync();
    const int e0 = int(me) * chunk, e1 = min(n_el, e0 + chunk);
    for (int idx = e0 + threadIdx.x; idx < e1; idx += kThreads) {
      const int row = idx / D, off = idx - e0;
      float lv[kMaxCluster], ov[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        lv[r] = r < ns ? rv_l[r * 16 + row] : -INFINITY;
        ov[r] = r < ns ? rv_o[r * chunk + off] : 0.f;
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (lv[r] < INFINITY) M = fmaxf(M, lv[r]);
      float acc = 0.f, tot = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (!(lv[r] > -INFINITY && lv[r] < INFINITY)) continue;   // an empty (or broken) partial
        const float w = ex2_approx((lv[r] - M) * kLog2e);
        acc = fmaf(w, ov[r], acc);
        tot += w;
      }
      reinterpret_cast<uint16_t*>(outp)[idx] = E::from_f(tot > 0.f ? acc * rcp_approx(tot) : 0.f);
      if (a.lse && idx % D == 0)
        a.lse[int64_t(b) * a.H_q + int64_t(h) * G + row] = tot > 0.f ? M + lg2_approx(tot) * kLn2 : -INFINITY;
    }
  } else {
  // ticket merge: partials to the workspace, the last CTA of the unit merges
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int row = idx / D;
    const int64_t pi = (int64_t(unit) * a.nsplit + split) * G + row;
    a.part_o[pi * D + idx % D] = merged(row, idx % D);
  }
  if (threadIdx.x < G) a.part_lse[(int64_t(unit) * a.nsplit + split) * G + threadIdx.x] = s_rl[threadIdx.x];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&a.tickets[unit], 1) == a.nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float* wgt = reinterpret_cast<float*>(smem);                // [nsplit][G]
  float* rmax = wgt + kMaxSplit * 16;                          // [G]
  float* rtot = rmax + 16;                                     // [G]
  const int64_t pbase = int64_t(unit) * a.nsplit * G;
  for (int i = threadIdx.x; i < a.nsplit * G; i += kThreads) {
    float v = __ldcg(a.part_lse + pbase + i);
    if (isinf(v)) v = -INFINITY;
    wgt[i] = v;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int row = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < a.nsplit; ++s) M = fmaxf(M, wgt[s * G + row]);
    rmax[row] = M;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.nsplit * G; i += kThreads) {
    const float M = rmax[i % G];
    const float v = wgt[i];
    wgt[i] = (M == -INFINITY || v == -INFINITY) ? 0.f : ex2_approx((v - M) * kLog2e);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int row = threadIdx.x;
    float t = 0.f;
    for (int s = 0; s < a.nsplit; ++s) t += wgt[s * G + row];
    rtot[row] = t > 0.f ? rcp_approx(t) : 0.f;
    if (a.lse)
      a.lse[int64_t(b) * a.H_q + int64_t(h) * G + row] =
          t > 0.f ? rmax[row] + lg2_approx(t) * kLn2 : -INFINITY;
  }
  __syncthreads();
  // every output element of the unit: sum over splits, loads issued 4 splits
  // at a time for all of this thread's elements before any is used
  constexpr int kOut = (16 * D) / kThreads;                    // elements per thread (G <= 16)
  const int n_el = G * D;
  float acc[kOut];
#pragma unroll
  for (int k = 0; k < kOut; ++k) acc[k] = 0.f;
  for (int s0 = 0; s0 < a.nsplit; s0 += 4) {
    float v[kOut][4];
#pragma unroll
    for (int k = 0; k < kOut; ++k) {
      const int idx = threadIdx.x + k * kThreads;
      const int row = idx / D, d = idx % D;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[k][u] = (idx < n_el && s0 + u < a.nsplit)
                      ? __ldcg(a.part_o + (pbase + int64_t(s0 + u) * G + row) * D + d)
                      : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kOut; ++k) {
      const int idx = threadIdx.x + k * kThreads;
      const int row = (idx < n_el ? idx : 0) / D;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (s0 + u < a.nsplit) {
          const float w = wgt[(s0 + u) * G + row];
          if (w != 0.f) acc[k] += w * v[k][u];
        }
    }
  }
#pragma unroll
  for (int k = 0; k < kOut; ++k) {
    const int idx = threadIdx.x + k * kThreads;
    if (idx < n_el) reinterpret_cast<uint16_t*>(outp)[idx] = E::from_f(acc[k] * rtot[idx / D]);
  }
  if (threadIdx.x == 0) a.tickets[unit] = 0;
  }  // ticket merge
}

// Splits per (request, KV head): one wave of resident CTAs, at most one split
// per tile, and enough splits that a CTA's entry table stays small.
int choose_nsplit(int units, int max_tiles, int ps, int sms) {
  const int target = kCtasPerSm * sms;
  int s = target / units;
  if (s > kMaxCluster) s = kMaxCluster;      // split CTAs of a unit fit one cluster
  const int64_t ent_total = (int64_t(max_tiles) * 16 + ps - 1) / ps;
  const int need = int((ent_total + kMaxEnt - 1) / kMaxEnt);
  if (s < need) s = need;
  if (s > max_tiles) s = max_tiles;
  if (s > kMaxSplit) s = kMaxSplit;
  return s < 1 ? 1 : s;
}

int ent_max_for(int max_tiles, int nsplit, int ps) {
  const int per = (max_tiles + nsplit - 1) / nsplit;
  return (per * 16 + ps - 1) / ps + 1;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t tickets, part_lse, part_o, total;
};

WsLayout ws_layout(int units, int G, int D, int nsplit) {
  WsLayout w;
  w.tickets = 0;
  w.part_lse = align256(size_t(units) * sizeof(int32_t));
  w.part_o = w.part_lse + align256(size_t(units) * nsplit * G * sizeof(float));
  w.total = w.part_o + align256(size_t(units) * nsplit * G * D * sizeof(float));
  return w;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);
EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// Tensor map over every pool row: [rows = num_blocks * H * page_size, D], box 16 x 64, 128-byte swizzle.
bool make_pool_map(CUtensorMap* m, const void* base, const sa_cache* c) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t rows = cuuint64_t(c->num_blocks) * c->num_kv_heads * c->page_size;
  if (rows >= (cuuint64_t(1) << 31)) return false;
  const cuuint64_t dims[2] = {cuuint64_t(c->head_dim), rows};
  const cuuint64_t strides[1] = {cuuint64_t(c->head_dim) * 2};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_dec_smem[16][64];

template <typename T, int D, bool kTma, bool kCluster>
sa_status launch_decode(const DecodeArgs& a, dim3 grid, cudaStream_t s, const CUtensorMap& mk,
                        const CUtensorMap& mv, int* cache, bool pdl) {
  auto k = decode_kernel<T, D, kTma, kCluster>;
  const int smem = kCluster ? recv_off(Tile<D>::kSmem, a.ent_max) + recv_bytes<D>()
                            : Tile<D>::kSmem + a.ent_max * int(sizeof(int2));
  if (!ensure_smem(k, smem, cache)) return SA_ERR_CUDA;
  const cudaError_t e = launch_ex(k, grid, dim3(kThreads), size_t(smem), s, pdl, kCluster ? grid.x : 1u,
                                  a, mk, mv);
  if (e == cudaSuccess) return SA_OK;
  if (!kCluster) return SA_ERR_CUDA;
  (void)cudaGetLastError();
  return SA_ERR_UNSUPPORTED;                     // caller falls back to the ticket merge
}

template <typename T, int D, bool kTma>
sa_status launch_merge_mode(const DecodeArgs& a, dim3 grid, cudaStream_t s, const CUtensorMap& mk,
                            const CUtensorMap& mv, int slot, bool allow_cluster, bool pdl) {
  if (allow_cluster && a.nsplit > 1 && a.nsplit <= kMaxCluster) {
    const sa_status st =
        launch_decode<T, D, kTma, true>(a, grid, s, mk, mv, g_dec_smem[4 * slot + 2 + kTma], pdl);
    if (st != SA_ERR_UNSUPPORTED) return st;
  }
  if (a.nsplit > 1 && !a.tickets && !a.logits_only) return SA_ERR_WORKSPACE;
  return launch_decode<T, D, kTma, false>(a, grid, s, mk, mv, g_dec_smem[4 * slot + kTma], pdl);
}

template <typename T, int D>
sa_status dispatch_tma(const DecodeArgs& a, dim3 grid, cudaStream_t s, const sa_cache* c, int slot,
                       bool allow_cluster, bool pdl) {
  CUtensorMap mk, mv;
  if (c->page_size >= 16 && make_pool_map(&mk, c->k, c) && make_pool_map(&mv, c->v, c))
    return launch_merge_mode<T, D, true>(a, grid, s, mk, mv, slot, allow_cluster, pdl);
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  return launch_merge_mode<T, D, false>(a, grid, s, mk, mv, slot, allow_cluster, pdl);
}

}  // namespace

sa_status decode_impl(const sa_cache* cache, const sa_batch* batch, const void* q, int32_t num_q_heads,
                      const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_stride, float scale,
                      void* out, float* lse, float* logits, int32_t logits_stride, void* workspace,
                      size_t workspace_bytes, int32_t* dev_status, void* stream, bool allow_cluster,
                      bool pdl, bool per_query_head, bool logits_only) {
  sa_status st = check_cache(cache, true, false);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (!q || !sel_idx || !sel_cnt || !out || sel_stride <= 0) return SA_ERR_INVALID_ARG;
  if (!aligned16(q)) return SA_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return SA_ERR_INVALID_ARG;
  const int G_kv = num_q_heads / cache->num_kv_heads;
  if (G_kv > 16) return SA_ERR_UNSUPPORTED;
  // per-query-head selection: every query head is its own unit of one row
  const int G = per_query_head ? 1 : G_kv;
  const int H_u = per_query_head ? num_q_heads : cache->num_kv_heads;
  const int64_t rows = int64_t(sel_stride) * cache->page_size;
  if (rows > (int64_t(1) << 30)) return SA_ERR_UNSUPPORTED;
  if (logits && logits_stride < rows) return SA_ERR_INVALID_ARG;
  const int units = batch->batch * H_u;
  const int max_tiles = int((rows + 15) / 16);
  const int ns = choose_nsplit(units, max_tiles, cache->page_size, sm_count());
  const WsLayout w = ws_layout(units, G, cache->head_dim, ns);
  if (logits_only && !logits) return SA_ERR_INVALID_ARG;
  if (ns > 1 && !logits_only && (!workspace || workspace_bytes < w.total)) return SA_ERR_WORKSPACE;
  DecodeArgs a;
  a.k = cache->k; a.v = cache->v; a.q = q; a.bt = batch->block_table; a.seq_lens = batch->seq_lens;
  a.sel = sel_idx; a.cnt = sel_cnt; a.out = out; a.lse = lse; a.logits = logits;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.tickets = ns > 1 ? reinterpret_cast<int32_t*>(ws + w.tickets) : nullptr;
  a.part_lse = ns > 1 ? reinterpret_cast<float*>(ws + w.part_lse) : nullptr;
  a.part_o = ns > 1 ? reinterpret_cast<float*>(ws + w.part_o) : nullptr;
  a.status = dev_status;
  a.H_kv = cache->num_kv_heads; a.H_q = num_q_heads; a.G = G; a.ps = cache->page_size;
  a.ps_shift = log2i(cache->page_size); a.num_blocks = cache->num_blocks;
  a.bt_stride = batch->bt_stride; a.sel_stride = sel_stride;
  a.logits_stride = logits ? logits_stride : 0; a.nsplit = ns;
  a.H_u = H_u; a.kv_div = per_query_head ? G_kv : 1;
  a.logits_only = logits_only ? 1 : 0;
  a.ent_max = ent_max_for(max_tiles, ns, cache->page_size);
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf(float(cache->head_dim));
  a.scale_log2 = a.scale * kLog2e;
  dim3 grid(unsigned(ns), unsigned(H_u), unsigned(batch->batch));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = cache->dtype == SA_BF16;
  if (cache->head_dim == 128)
    return bf ? dispatch_tma<__nv_bfloat16, 128>(a, grid, s, cache, 0, allow_cluster, pdl)
              : dispatch_tma<__half, 128>(a, grid, s, cache, 1, allow_cluster, pdl);
  return bf ? dispatch_tma<__nv_bfloat16, 64>(a, grid, s, cache, 2, allow_cluster, pdl)
            : dispatch_tma<__half, 64>(a, grid, s, cache, 3, allow_cluster, pdl);
}

}  // namespace sa

extern "C" size_t sa_decode_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t num_q_heads,
                                           int32_t head_dim, int32_t page_size, int32_t sel_stride) {
  using namespace sa;
  if (batch <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      sel_stride <= 0 || num_q_heads % num_kv_heads)
    return 0;
  const int units = batch * num_kv_heads;
  const int64_t max_tiles = (int64_t(sel_stride) * page_size + 15) / 16;
  const int ns = choose_nsplit(units, int(max_tiles > (1 << 30) ? (1 << 30) : max_tiles), page_size,
                               sm_count());
  return ws_layout(units, num_q_heads / num_kv_heads, head_dim, ns).total;
}

extern "C" sa_status sa_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes == 0) return SA_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

extern "C" sa_status sa_sparse_decode(const sa_cache* cache, const sa_batch* batch, const void* q,
                                      int32_t num_q_heads, const int32_t* sel_idx,
                                      const int32_t* sel_cnt, int32_t sel_stride, float scale,
                                      void* out, float* lse, float* logits, int32_t logits_stride,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                      void* stream) {
  return sa::decode_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, sel_stride, scale, out, lse,
                         logits, logits_stride, workspace, workspace_bytes, dev_status, stream, true, false,
                         false, false);
}

extern "C" sa_status sa_sparse_decode_qh(const sa_cache* cache, const sa_batch* batch, const void* q,
                                         int32_t num_q_heads, const int32_t* sel_idx,
                                         const int32_t* sel_cnt, int32_t sel_stride, float scale,
                                         void* out, float* lse, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return sa::decode_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, sel_stride, scale, out, lse,
                         nullptr, 0, workspace, workspace_bytes, dev_status, stream, true, false,
                         true, false);
}

// ---------------------------------------------------------------------------
// sa_sparse_decode_noalloc: the same split-K decode, with its scratch (split
// partials and per-(request, KV head) tickets) in a fixed device array of this
// library instead of a caller workspace, for callers that cannot allocate.
// ---------------------------------------------------------------------------
#ifndef SA_NOALLOC_SCRATCH_BYTES
#define SA_NOALLOC_SCRATCH_BYTES (4u << 20)
#endif

// Lives in every GPU that loads the library until the process exits. In host
// code this name is only a stand-in: the device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SA_NOALLOC_SCRATCH_BYTES];

namespace {
void* g_noalloc_addr[64];   // device address of g_noalloc_scratch, per device ordinal
}  // namespace

extern "C" size_t sa_sparse_decode_noalloc_capacity(void) { return SA_NOALLOC_SCRATCH_BYTES; }

extern "C" sa_status sa_sparse_decode_noalloc(const sa_cache* cache, const sa_batch* batch,
                                              const void* q, int32_t num_q_heads,
                                              const int32_t* sel_idx, const int32_t* sel_cnt,
                                              int32_t sel_stride, float scale, void* out, float* lse,
                                              float* logits, int32_t logits_stride,
                                              int32_t* dev_status, void* stream) {
  using namespace sa;
  if (!cache || !batch || cache->num_kv_heads <= 0 || num_q_heads <= 0 || sel_stride <= 0 ||
      num_q_heads % cache->num_kv_heads || cache->head_dim <= 0 || cache->page_size <= 0 ||
      batch->batch <= 0)
    return SA_ERR_INVALID_ARG;
  const size_t need = sa_decode_workspace_size(batch->batch, cache->num_kv_heads, num_q_heads,
                                               cache->head_dim, cache->page_size, sel_stride);
  if (need == 0) return SA_ERR_INVALID_ARG;
  if (need > SA_NOALLOC_SCRATCH_BYTES) return SA_ERR_WORKSPACE;   // beyond the fixed scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SA_ERR_CUDA;
  if (!g_noalloc_addr[dev]) {
    // set-up on this device's first call (do it before any stream capture)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  void* ws = g_noalloc_addr[dev];
  // the tickets must start at zero on every call (a call cut short could leave them set)
  const size_t ticket_bytes = size_t(batch->batch) * cache->num_kv_heads * sizeof(int32_t);
  if (cudaMemsetAsync(ws, 0, ticket_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SA_ERR_CUDA;
  return sa::decode_impl(cache, batch, q, num_q_heads, sel_idx, sel_cnt, sel_stride, scale, out, lse,
                         logits, logits_stride, ws, SA_NOALLOC_SCRATCH_BYTES, dev_status, stream,
                         /*allow_cluster=*/false, /*pdl=*/false, /*per_query_head=*/false,
                         /*logits_only=*/false);
}
