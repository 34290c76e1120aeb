// Status strings and version of the C ABI.
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
