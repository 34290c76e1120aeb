// Status strings and version of the C ABI, and the self-test of the bounded
// in-kernel wait every kernel of the library uses.
#include "common.cuh"
#include "sparse_attn.h"

extern "C" const char* sa_status_string(sa_status status) {
  switch (status) {
    case SA_OK: return "SA_OK";
    case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
    case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED";
    case SA_ERR_WORKSPACE: return "SA_ERR_WORKSPACE";
    case SA_ERR_CUDA: return "SA_ERR_CUDA";
  }
  return "SA_ERR_UNKNOWN";
}

extern "C" const char* sa_version(void) { return "0.1.0"; }

extern "C" size_t sa_struct_size(int32_t which) {
  return which == 0 ? sizeof(sa_cache) : (which == 1 ? sizeof(sa_batch) : 0);
}

namespace sa {
namespace {

// One warp waits on an mbarrier that expects two arrivals and receives
// `arrivals` of them, through the same bounded wait the library's kernels use.
__global__ void wait_selftest_kernel(int arrivals, uint64_t limit_ns, int32_t* status, int32_t* result) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 2);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int i = 0; i < arrivals; ++i) mbar_arrive(b);
  __syncwarp();
  const bool ok = mbar_wait(b, 0, status, limit_ns);
  if (threadIdx.x == 0) *result = ok ? 1 : 0;
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_wait_selftest(int32_t arrivals, int64_t limit_ns, int32_t* dev_status,
                                      int32_t* result, void* stream) {
  if (!dev_status || !result || arrivals < 0 || arrivals > 2) return SA_ERR_INVALID_ARG;
  if (limit_ns <= 0 || limit_ns > 100000000) return SA_ERR_INVALID_ARG;
  sa::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      arrivals, uint64_t(limit_ns), dev_status, result);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}
