// sa_h2o_prefill: H2O absorb and eviction for incoming tokens, each token's
// own key standing in for its query.
//
// "H2O -- Cumulative Attention-Mass Heavy-Hitter Oracle Eviction"
// (VeloxQuant-MLX), "How it works": for every incoming token (prefill and
// decode), per head, the new key attends to every stored key (scaled
// softmax), the stored scores decay and take that attention, the new token
// starts at 0, and above budget the lowest-scoring entry outside the first
// n_sink and the newest grace entries is removed (first index on a tie: the
// lowest position). The changelog's batched absorb of a below-budget prefix is
// the same arithmetic as this token-by-token loop. Scores are held in bf16 and
// each fold is one float64 fma rounded once, as in sa_h2o_update.
//
// One CTA (512 threads) per (KV head, request) runs the request's new tokens
// in order. The retained keys stay in shared memory for the whole call (rows
// padded by 16 bytes so a warp's rows fall in different bank groups), held in
// slots that are reused when an entry leaves; `order` lists the slots by
// position, so the protected windows are list indices as in the decode-side
// update. At the end the list, scores and evicted positions go back to memory.
#include "common.cuh"
#include "host.h"

namespace sa {
namespace {

constexpr int kPxThreads = 512;
constexpr int kPxWarps = kPxThreads / 32;
constexpr int kPxSmemLimit = 200 * 1024;

struct ProxyArgs {
  const uint16_t* k;            // pool [num_blocks, H, 1, D]
  const int32_t* bt;
  const int32_t* seq_lens;
  const int32_t* new_cu;
  uint16_t* hh;                 // [num_slots, H] bf16
  int32_t* ret_pos;
  int32_t* ret_cnt;
  int32_t* evicted;
  int32_t* evicted_cnt;
  int32_t* status;
  int H, bt_stride, num_blocks, cap, ev_cap, budget, n_sink, grace, slots;
  float decay, scale;
};

template <int D>
struct PxLayout {
  static constexpr int kRow = (D + 8) * 2;   // bytes of a padded key row
  // key rows | positions | scores | order | the new key as float (16-byte aligned)
  static __host__ __device__ int kf_off(int slots) { return (slots * (kRow + 12) + 15) & ~15; }
  static __host__ __device__ int bytes(int slots) { return kf_off(slots) + D * 4; }
};

__device__ __forceinline__ float block_max_f(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = lane < kPxWarps ? red[lane] : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(kFull, r, o));
  __syncthreads();
  return r;
}

__device__ __forceinline__ float block_sum_f(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = lane < kPxWarps ? red[lane] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(kFull, r, o);
  __syncthreads();
  return r;
}

__device__ __forceinline__ uint64_t block_min_u64(uint64_t v, uint64_t* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t y = __shfl_xor_sync(kFull, v, o);
    v = y < v ? y : v;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint64_t r = lane < kPxWarps ? red[lane] : ~0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t y = __shfl_xor_sync(kFull, r, o);
    r = y < r ? y : r;
  }
  __syncthreads();
  return r;
}

template <int D>
__global__ void __launch_bounds__(kPxThreads) h2o_proxy_kernel(ProxyArgs a) {
  using L = PxLayout<D>;
  extern __shared__ __align__(16) uint8_t sm[];
  const int S = a.slots;                                   // budget + 1
  uint8_t* krow = sm;                                      // [S][D + 8] bf16
  int32_t* s_pos = reinterpret_cast<int32_t*>(sm + S * L::kRow);
  float* s_hh = reinterpret_cast<float*>(s_pos + S);
  int32_t* order = reinterpret_cast<int32_t*>(s_hh + S);   // slots by position
  float* s_kf = reinterpret_cast<float*>(sm + L::kf_off(S));   // the new key, float [D]
  __shared__ float red[kPxWarps];
  __shared__ uint64_t redu[kPxWarps];
  __shared__ int s_slot;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int unit = b * a.H + h;
  const int Lnew = a.seq_lens[b];
  const int n_new = a.new_cu[b + 1] - a.new_cu[b];
  const int L0 = Lnew - n_new;                             // positions L0 .. Lnew-1 arrive
  int cnt = a.ret_cnt[unit];
  if (cnt < 0 || cnt > a.budget) {
    if (tid == 0) flag(a.status, SA_DEV_BAD_COUNT);
    cnt = cnt < 0 ? 0 : a.budget;
  }
  if (n_new < 0 || L0 < 0 || Lnew > a.bt_stride) {
    if (tid == 0) flag(a.status, SA_DEV_OVERFLOW);
    return;
  }
  int32_t* rp = a.ret_pos + int64_t(unit) * a.cap;
  int bad = 0;

  // the retained entries into slots 0 .. cnt-1 (list order = slot order at first)
  for (int j = tid; j < cnt; j += kPxThreads) {
    const int pos = rp[j];
    int blk = (pos >= 0 && pos < a.bt_stride) ? a.bt[int64_t(b) * a.bt_stride + pos] : -1;
    if (blk < 0 || blk >= a.num_blocks) { flag(a.status, SA_DEV_BAD_BLOCK); blk = -1; }
    s_pos[j] = pos;
    order[j] = j;
    s_hh[j] = blk >= 0 ? Elem<__nv_bfloat16>::to_f(a.hh[int64_t(blk) * a.H + h]) : 0.f;
    bad |= blk < 0;
  }
  for (int idx = tid; idx < cnt * (D / 8); idx += kPxThreads) {
    const int j = idx / (D / 8), c = idx % (D / 8);
    const int pos = rp[j];                                 // (s_pos[j] is another thread's write)
    const int blk = (pos >= 0 && pos < a.bt_stride) ? a.bt[int64_t(b) * a.bt_stride + pos] : -1;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (blk >= 0 && blk < a.num_blocks)
      v = *reinterpret_cast<const uint4*>(a.k + (int64_t(blk) * a.H + h) * D + c * 8);
    *reinterpret_cast<uint4*>(krow + j * L::kRow + c * 16) = v;
  }
  if (__syncthreads_or(bad)) return;                       // a bad block: the unit is left as it was

  int next_slot = cnt, free_slot = -1, n_ev = 0;
  const double decay = double(a.decay);
  for (int t = 0; t < n_new; ++t) {
    const int pos_new = L0 + t;
    const int blk_new = a.bt[int64_t(b) * a.bt_stride + pos_new];
    if (blk_new < 0 || blk_new >= a.num_blocks) {           // uniform across the CTA
      if (tid == 0) flag(a.status, SA_DEV_BAD_BLOCK);
      break;
    }
    const int slot = free_slot >= 0 ? free_slot : next_slot;
    // the new key: float copy for the dot products, raw row into its slot
    if (tid < D / 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(a.k + (int64_t(blk_new) * a.H + h) * D + tid * 8);
      *reinterpret_cast<uint4*>(krow + slot * L::kRow + tid * 16) = v;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s_kf[tid * 8 + 2 * e] = Elem<__nv_bfloat16>::lo(w[e]);
        s_kf[tid * 8 + 2 * e + 1] = Elem<__nv_bfloat16>::hi(w[e]);
      }
    }
    __syncthreads();
    if (cnt > 0) {
      // attention of the new key over the stored ones (list index j, slot order[j])
      float z[2] = {-INFINITY, -INFINITY};                  // budget + 1 <= 2 * 512
      float m = -INFINITY;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = tid + r * kPxThreads;
        if (j < cnt) {
          const uint8_t* row = krow + order[j] * L::kRow;
          float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
          for (int c = 0; c < D / 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + c * 16);
            const float4 q0 = *reinterpret_cast<const float4*>(s_kf + c * 8);
            const float4 q1 = *reinterpret_cast<const float4*>(s_kf + c * 8 + 4);
            acc0 = fmaf(Elem<__nv_bfloat16>::lo(v.x), q0.x, acc0);
            acc1 = fmaf(Elem<__nv_bfloat16>::hi(v.x), q0.y, acc1);
            acc0 = fmaf(Elem<__nv_bfloat16>::lo(v.y), q0.z, acc0);
            acc1 = fmaf(Elem<__nv_bfloat16>::hi(v.y), q0.w, acc1);
            acc0 = fmaf(Elem<__nv_bfloat16>::lo(v.z), q1.x, acc0);
            acc1 = fmaf(Elem<__nv_bfloat16>::hi(v.z), q1.y, acc1);
            acc0 = fmaf(Elem<__nv_bfloat16>::lo(v.w), q1.z, acc0);
            acc1 = fmaf(Elem<__nv_bfloat16>::hi(v.w), q1.w, acc1);
          }
          z[r] = (acc0 + acc1) * a.scale;
          m = fmaxf(m, z[r]);
        }
      }
      m = block_max_f(m, red);
      float e[2] = {0.f, 0.f}, sum = 0.f;
#pragma unroll
      for (int r = 0; r < 2; ++r)
        if (tid + r * kPxThreads < cnt) { e[r] = expf(z[r] - m); sum += e[r]; }
      sum = block_sum_f(sum, red);
      const float inv = 1.0f / sum;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = tid + r * kPxThreads;
        if (j < cnt) {
          const int sl = order[j];
          const uint16_t nb = round_f64<8, -126, 127>(fma(decay, double(s_hh[sl]), double(e[r] * inv)));
          s_hh[sl] = Elem<__nv_bfloat16>::to_f(nb);
        }
      }
    }
    // the new token enters at the end of the list with score 0
    if (tid == 0) {
      order[cnt] = slot;
      s_pos[slot] = pos_new;
      s_hh[slot] = 0.f;
    }
    if (free_slot >= 0) free_slot = -1; else ++next_slot;
    ++cnt;
    __syncthreads();
    if (cnt > a.budget) {
      // the eligible entry with the least (score, position); scores are >= 0,
      // so their bf16 bits order like their values
      const int lo = a.n_sink, hi = cnt - a.grace;
      uint64_t best = ~0ull;
      for (int j = lo + tid; j < hi; j += kPxThreads) {
        const int sl = order[j];
        const uint32_t bits = __float_as_uint(s_hh[sl]) >> 16;
        const uint64_t key = (uint64_t(bits) << 32) | uint32_t(s_pos[sl]);
        best = key < best ? key : best;
      }
      best = block_min_u64(best, redu);
      const int pos_ev = int(uint32_t(best & 0xffffffffu));
      // its list index: the unique j in [lo, hi) holding pos_ev
      for (int j = lo + tid; j < hi; j += kPxThreads)
        if (s_pos[order[j]] == pos_ev) s_slot = j;
      __syncthreads();
      const int jev = s_slot;
      free_slot = order[jev];
      if (tid == 0 && a.evicted && n_ev < a.ev_cap) a.evicted[int64_t(unit) * a.ev_cap + n_ev] = pos_ev;
      if (n_ev >= a.ev_cap && tid == 0 && a.evicted) flag(a.status, SA_DEV_OVERFLOW);
      ++n_ev;
      // close the gap in the list
      int mv[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = jev + tid + r * kPxThreads;
        mv[r] = j + 1 < cnt ? order[j + 1] : 0;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = jev + tid + r * kPxThreads;
        if (j + 1 < cnt) order[j] = mv[r];
      }
      --cnt;
      __syncthreads();
    }
  }

  // back to memory: the list in position order, its scores, the counts
  for (int j = tid; j < cnt; j += kPxThreads) {
    const int sl = order[j];
    const int pos = s_pos[sl];
    rp[j] = pos;
    const int blk = a.bt[int64_t(b) * a.bt_stride + pos];
    if (blk >= 0 && blk < a.num_blocks)
      a.hh[int64_t(blk) * a.H + h] = uint16_t(__float_as_uint(s_hh[sl]) >> 16);
  }
  if (tid == 0) {
    a.ret_cnt[unit] = cnt;
    if (a.evicted_cnt) a.evicted_cnt[unit] = min(n_ev, a.ev_cap);
  }
}

int g_px_smem[2][64];

template <int D>
sa_status launch_proxy(const ProxyArgs& a, dim3 grid, cudaStream_t s, int* attr) {
  const int smem = PxLayout<D>::bytes(a.slots);
  if (smem > kPxSmemLimit) return SA_ERR_UNSUPPORTED;
  if (!ensure_smem(h2o_proxy_kernel<D>, smem, attr)) return SA_ERR_CUDA;
  h2o_proxy_kernel<D><<<grid, kPxThreads, smem, s>>>(a);
  return launch_status();
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_h2o_prefill(const sa_cache* cache, const sa_batch* batch,
                                    const int32_t* new_cu, void* hh, int32_t num_slots,
                                    int32_t* ret_pos, int32_t* ret_cnt, int32_t ret_cap,
                                    int32_t budget, int32_t n_sink, int32_t grace, float decay,
                                    float scale, int32_t* evicted, int32_t* evicted_cnt,
                                    int32_t evicted_cap, int32_t* dev_status, void* stream) {
  using namespace sa;
  sa_status st = check_cache(cache, true, false);
  if (st != SA_OK) return st;
  if ((st = check_batch(batch)) != SA_OK) return st;
  if (cache->page_size != 1 || cache->dtype != SA_BF16) return SA_ERR_UNSUPPORTED;
  if (!new_cu || !hh || !ret_pos || !ret_cnt || num_slots <= 0) return SA_ERR_INVALID_ARG;
  if (ret_cap <= 0 || budget <= 0 || budget > ret_cap) return SA_ERR_INVALID_ARG;
  if (n_sink < 0 || grace < 0 || budget <= n_sink + grace) return SA_ERR_INVALID_ARG;
  if (!(decay > 0.f && decay <= 1.f)) return SA_ERR_INVALID_ARG;
  if ((evicted == nullptr) != (evicted_cnt == nullptr) || (evicted && evicted_cap <= 0))
    return SA_ERR_INVALID_ARG;
  if (budget + 1 > 2 * kPxThreads) return SA_ERR_UNSUPPORTED;
  ProxyArgs a;
  a.k = static_cast<const uint16_t*>(cache->k); a.bt = batch->block_table; a.seq_lens = batch->seq_lens;
  a.new_cu = new_cu; a.hh = static_cast<uint16_t*>(hh); a.ret_pos = ret_pos; a.ret_cnt = ret_cnt;
  a.evicted = evicted; a.evicted_cnt = evicted_cnt; a.status = dev_status;
  a.H = cache->num_kv_heads; a.bt_stride = batch->bt_stride; a.num_blocks = cache->num_blocks;
  a.cap = ret_cap; a.ev_cap = evicted ? evicted_cap : 0; a.budget = budget; a.n_sink = n_sink;
  a.grace = grace; a.slots = budget + 1; a.decay = decay;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf(float(cache->head_dim));
  dim3 grid(unsigned(cache->num_kv_heads), unsigned(batch->batch));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cache->head_dim == 128 ? launch_proxy<128>(a, grid, s, g_px_smem[0])
                                : launch_proxy<64>(a, grid, s, g_px_smem[1]);
}
