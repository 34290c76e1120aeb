// Host-side helpers shared by the C-ABI entry points: argument checks and
// per-device kernel attribute setup.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_attn.h"

namespace sa {

inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

inline int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

inline sa_status check_cache(const sa_cache* c, bool need_kv, bool need_meta) {
  if (!c) return SA_ERR_INVALID_ARG;
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

inline sa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

// Raise a kernel's dynamic shared-memory limit on the current device once.
template <typename K>
inline bool ensure_smem(K kernel, int bytes, int* cache_per_device) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (cache_per_device[dev] >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  cache_per_device[dev] = bytes;
  return true;
}

}  // namespace sa
