// Host-side helpers shared by the C-ABI entry points: argument checks and
// per-device kernel attribute setup.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "sparse_attn.h"

namespace sa {

inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

inline int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

// vector loads and bulk copies read whole 16-byte units
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline sa_status check_cache(const sa_cache* c, bool need_kv, bool need_meta) {
  if (!c) return SA_ERR_INVALID_ARG;
  if (!aligned16(c->k) || !aligned16(c->v) || !aligned16(c->meta) || !aligned16(c->kstd))
    return SA_ERR_INVALID_ARG;
  if (c->dtype != SA_BF16 && c->dtype != SA_FP16) return SA_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0) return SA_ERR_INVALID_ARG;
  if (!is_pow2(c->page_size) || c->page_size > 128) return SA_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return SA_ERR_UNSUPPORTED;
  if (need_kv && (!c->k || !c->v)) return SA_ERR_INVALID_ARG;
  if (need_meta && !c->meta) return SA_ERR_INVALID_ARG;
  return SA_OK;
}

inline sa_status check_batch(const sa_batch* b) {
  if (!b || !b->block_table || !b->seq_lens) return SA_ERR_INVALID_ARG;
  if (b->batch <= 0 || b->bt_stride <= 0) return SA_ERR_INVALID_ARG;
  return SA_OK;
}

// SMs of the current device (cached per device; 148 if it cannot be read)
inline int sm_count() {
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

inline sa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

// Raise a kernel's dynamic shared-memory limit on the current device once, and
// ask for the largest shared-memory carveout. Every kernel of a step asks for
// the same carveout, so a kernel launched programmatically beside another can
// take free slots on an SM without waiting for it to drain and reconfigure.
// cache_per_device[dev] holds the bytes already set plus one.
template <typename K>
inline bool ensure_smem(K kernel, int bytes, int* cache_per_device) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (cache_per_device[dev] > bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
    return false;
  cache_per_device[dev] = bytes + 1;
  return true;
}

// Launch with optional programmatic dependent launch (the kernel may start
// before its predecessor in the stream completes; it must call pdl_wait()
// before touching anything the predecessor writes) and optional cluster size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, bool pdl, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Internal entry points shared by the public calls and the fused step.
sa_status append_impl(const sa_cache* cache, const sa_batch* batch, const void* k_new,
                      const void* v_new, const int32_t* new_cu, int32_t max_new_per_req, void* hh,
                      int32_t* ret_pos, int32_t* ret_cnt, int32_t ret_cap, int32_t* dev_status,
                      void* stream, bool pdl);
sa_status score_impl(const sa_cache* cache, const sa_batch* batch, const void* q, int32_t num_q_heads,
                     float w_avg, float w_peak, float* scores, int32_t max_pages, int32_t* dev_status,
                     void* stream, bool per_query_head);
sa_status select_impl(const float* scores, int32_t max_pages, const sa_batch* batch, int32_t page_size,
                      int32_t num_kv_heads, int32_t topk, int32_t n_bos, int32_t n_eos,
                      int32_t* sel_idx, int32_t* sel_cnt, int32_t* dev_status, void* stream,
                      bool pdl);
sa_status decode_impl(const sa_cache* cache, const sa_batch* batch, const void* q, int32_t num_q_heads,
                      const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_stride, float scale,
                      void* out, float* lse, float* logits, int32_t logits_stride, void* workspace,
                      size_t workspace_bytes, int32_t* dev_status, void* stream, bool allow_cluster,
                      bool pdl, bool per_query_head, bool logits_only = false);

}  // namespace sa
