// Shared device helpers of the sm_103a sparse-decode kernels: element types,
// exact rounding from float64, inline-PTX wrappers (cp.async, ldmatrix,
// mma.sync, non-coherent vector loads) and small block-wide scans.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_attn.h"

namespace sa {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void flag(int32_t* status, int bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------------------
// IEEE 754 round-to-nearest-even of a float64 onto a narrower binary format
// with P significand bits and normal exponents [EMIN, EMAX] (bias = EMAX).
// One rounding straight from the float64 value (no float32 intermediate).
// Written from the format definition: drop the low significand bits, round
// half to even, carry into the next binade, saturate to infinity, and use the
// fixed subnormal spacing 2^(EMIN-P+1) below the smallest normal.
// ---------------------------------------------------------------------------
template <int P, int EMIN, int EMAX>
__device__ __forceinline__ uint16_t round_f64(double x) {
  constexpr int MB = P - 1;                  // stored significand bits
  constexpr int EB = 15 - MB;                // exponent bits
  constexpr uint16_t INF = uint16_t(((1u << EB) - 1u) << MB);
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(x));
  const uint16_t sign = uint16_t((u >> 63) << 15);
  const uint64_t a = u & 0x7fffffffffffffffull;
  if (a >= 0x7ff0000000000000ull) {          // inf / nan
    if (a > 0x7ff0000000000000ull) return uint16_t(sign | INF | (1u << (MB - 1)));
    return uint16_t(sign | INF);
  }
  if ((a >> 52) == 0) return sign;           // zero or float64 subnormal: far below half a quantum
  int e = int(a >> 52) - 1023;
  const uint64_t m = (a & 0x000fffffffffffffull) | (1ull << 52);
  int shift = 52 - MB;
  const bool sub = e < EMIN;
  if (sub) shift += EMIN - e;
  if (shift > 53) return sign;               // below half the smallest subnormal
  uint64_t r = m >> shift;
  const uint64_t rem = m & ((1ull << shift) - 1ull);
  const uint64_t half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (r & 1ull))) r += 1ull;
  if (sub) return uint16_t(sign | uint16_t(r));   // r == 2^MB encodes the smallest normal
  if (r >> P) { r >>= 1; e += 1; }
  if (e > EMAX) return uint16_t(sign | INF);
  return uint16_t(sign | uint16_t((e + EMAX) << MB) | uint16_t(r & ((1u << MB) - 1u)));
}

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
  static __device__ __forceinline__ float hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
  static __device__ __forceinline__ float to_f(uint16_t u) { return __uint_as_float(uint32_t(u) << 16); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
  }
  static __device__ __forceinline__ uint16_t from_f(float a) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(a));
  }
  static __device__ __forceinline__ uint16_t from_f64(double x) { return round_f64<8, -126, 127>(x); }
  static __device__ __forceinline__ uint16_t from_f_rz(float a) {
    return __bfloat16_as_ushort(__float2bfloat16_rz(a));
  }
  // 1: a float32 q lies exactly half-way between two bf16 values; 0: it does not;
  // -1: not decidable here (outside the range handled in float32).
  static __device__ __forceinline__ int midpoint(float q) {
    return (__float_as_uint(q) & 0xffffu) == 0x8000u ? 1 : 0;
  }
  static __device__ __forceinline__ void mma(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

template <>
struct Elem<__half> {
  static __device__ __forceinline__ float lo(uint32_t u) {
    return __half2float(__ushort_as_half(uint16_t(u & 0xffffu)));
  }
  static __device__ __forceinline__ float hi(uint32_t u) {
    return __half2float(__ushort_as_half(uint16_t(u >> 16)));
  }
  static __device__ __forceinline__ float to_f(uint16_t u) { return __half2float(__ushort_as_half(u)); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
  }
  static __device__ __forceinline__ uint16_t from_f(float a) {
    return __half_as_ushort(__float2half_rn(a));
  }
  static __device__ __forceinline__ uint16_t from_f64(double x) { return round_f64<11, -14, 15>(x); }
  static __device__ __forceinline__ uint16_t from_f_rz(float a) {
    return __half_as_ushort(__float2half_rz(a));
  }
  static __device__ __forceinline__ int midpoint(float q) {
    const float aq = fabsf(q);
    if (!(aq >= 0x1p-14f && aq <= 65504.f)) return -1;          // fp16 subnormal / overflow range
    return (__float_as_uint(q) & 0x1fffu) == 0x1000u ? 1 : 0;
  }
  static __device__ __forceinline__ void mma(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

// ---------------------------------------------------------------------------
// memory helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 zero-fills without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// ---------------------------------------------------------------------------
// mbarrier + bulk (TMA engine) copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of an mbarrier, giving up after limit_ns of wall
// time (~1 s by default; sets SA_DEV_TIMEOUT and returns false). Correct code
// never times out.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) {
      flag(status, SA_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Bulk copy global -> this CTA's shared memory, completion counted in bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled TMA load (tensor map in kernel-parameter space), completion on `bar`.
// x (innermost coordinate) * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Order this thread's generic-proxy shared-memory accesses before later async-proxy (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---------------------------------------------------------------------------
// programmatic dependent launch (no-ops unless the launch asked for it)
// ---------------------------------------------------------------------------
// Let the next kernel in the stream, if launched programmatically, start now.
// The SFU's approximate base-2 exponential, base-2 logarithm and reciprocal
// (single PTX instructions; subnormal results and inputs flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
// Wait until the grids this one depends on have completed and their memory is visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// ---------------------------------------------------------------------------
// thread-block clusters: rank, distributed shared memory, barrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// All threads of all CTAs of the cluster; release our shared-memory writes, acquire the others'.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The two halves of a cluster barrier phase, for a phase whose arrive is
// issued long before its wait (no memory ordering on the arrive).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(addr), "f"(v) : "memory");
}

// ---------------------------------------------------------------------------
// order-preserving keys
// ---------------------------------------------------------------------------
// float32 -> uint32 whose unsigned order is the float order, -0 == +0, NaN
// below every number (so a descending selection ranks it last).
__device__ __forceinline__ uint32_t f32_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// bf16 bits -> uint16 key in value order, -0 == +0, NaN above every number.
__device__ __forceinline__ uint32_t bf16_key(uint16_t u) {
  if ((u & 0x7fffu) > 0x7f80u) return 0xffffu;
  if (u == 0x8000u) u = 0;
  return (u & 0x8000u) ? (~uint32_t(u) & 0xffffu) : (uint32_t(u) | 0x8000u);
}

// Histogram increment aggregated across the warp: lanes holding the same bin
// add once (one shared-memory atomic per distinct bin per warp). Every lane of
// the warp must call it; `bin` < 0 means "no key on this lane".
__device__ __forceinline__ void warp_hist_add(int* hist, int bin) {
  const unsigned peers = __match_any_sync(kFull, bin);
  const int leader = __ffs(peers) - 1;
  if (bin >= 0 && (threadIdx.x & 31) == leader) atomicAdd(&hist[bin], __popc(peers));
}

// ---------------------------------------------------------------------------
// block-wide exclusive prefix sum of one int per thread (NT threads).
// `scratch` holds >= 32 ints. Returns the exclusive prefix; *total = sum.
// ---------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NT / 32 ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  const int before = (warp ? scratch[warp - 1] : 0) + x - v;
  *total = scratch[NT / 32 - 1];
  __syncthreads();
  return before;
}

}  // namespace sa
