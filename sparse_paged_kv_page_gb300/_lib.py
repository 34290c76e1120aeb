"""ctypes loader of the native library and the C struct mirrors.

Fails loudly when the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_sparse_attn.so")

c_i32 = ctypes.c_int32
c_ptr = ctypes.c_void_p
c_f32 = ctypes.c_float
c_size = ctypes.c_size_t

SA_BF16, SA_FP16 = 0, 1
SA_DEV_BAD_BLOCK, SA_DEV_OVERFLOW, SA_DEV_BAD_COUNT, SA_DEV_TIMEOUT = 1, 2, 4, 8


class SaCache(ctypes.Structure):
    _fields_ = [("k", c_ptr), ("v", c_ptr), ("meta", c_ptr), ("dtype", c_i32),
                ("num_blocks", c_i32), ("num_kv_heads", c_i32), ("page_size", c_i32),
                ("head_dim", c_i32), ("kstd", c_ptr)]


class SaBatch(ctypes.Structure):
    _fields_ = [("block_table", c_ptr), ("seq_lens", c_ptr), ("batch", c_i32),
                ("bt_stride", c_i32)]


P_CACHE = ctypes.POINTER(SaCache)
P_BATCH = ctypes.POINTER(SaBatch)

# name -> (restype, argtypes), as declared in include/sparse_attn.h
SIGNATURES = {
    "sa_append_kv": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr, c_ptr,
                             c_i32, c_ptr, c_ptr]),
    "sa_score_pages": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_f32, c_f32, c_ptr, c_i32,
                               c_ptr, c_ptr]),
    "sa_select_topk": (c_i32, [c_ptr, c_i32, P_BATCH, c_i32, c_i32, c_i32, c_ptr, c_ptr, c_ptr,
                               c_ptr]),
    "sa_decode_workspace_size": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "sa_decode_workspace_init": (c_i32, [c_ptr, c_size, c_ptr]),
    "sa_sparse_decode": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_f32,
                                 c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_size, c_ptr, c_ptr]),
    "sa_sparse_decode_noalloc": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_f32,
                                         c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr]),
    "sa_sparse_decode_noalloc_capacity": (c_size, []),
    "sa_h2o_update": (c_i32, [P_BATCH, c_i32, c_i32, c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_ptr,
                              c_ptr, c_i32, c_i32, c_i32, c_i32, c_f32, c_ptr, c_ptr, c_ptr,
                              c_ptr]),
    "sa_decode_step": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_i32, c_f32,
                               c_f32, c_ptr, c_i32, c_i32, c_i32, c_i32, c_ptr, c_ptr, c_f32,
                               c_ptr, c_ptr, c_ptr, c_size, c_ptr, c_ptr]),
    "sa_select_topk_reserved": (c_i32, [c_ptr, c_i32, P_BATCH, c_i32, c_i32, c_i32, c_i32, c_i32,
                                        c_ptr, c_ptr, c_ptr, c_ptr]),
    "sa_h2o_update_window": (c_i32, [P_BATCH, c_i32, c_i32, c_ptr, c_i32, c_ptr, c_ptr, c_i32,
                                     c_ptr, c_ptr, c_i32, c_i32, c_i32, c_i32, c_f32, c_ptr,
                                     c_ptr, c_ptr, c_ptr]),
    "sa_score_pages_qh": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_f32, c_f32, c_ptr, c_i32,
                                  c_ptr, c_ptr]),
    "sa_sparse_decode_qh": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_f32,
                                    c_ptr, c_ptr, c_ptr, c_size, c_ptr, c_ptr]),
    "sa_h2o_prefill": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_i32,
                               c_i32, c_i32, c_f32, c_f32, c_ptr, c_ptr, c_i32, c_ptr, c_ptr]),
    "sa_entmax_workspace_size": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "sa_sparse_decode_entmax": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_f32,
                                        c_f32, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_size, c_ptr,
                                        c_ptr]),
    "sa_sparse_decode_entmax_qh": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_ptr, c_ptr, c_i32,
                                           c_f32, c_f32, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_size,
                                           c_ptr, c_ptr]),
    "sa_gauss_select": (c_i32, [P_CACHE, P_BATCH, c_ptr, c_i32, c_f32, c_f32, c_ptr, c_i32, c_ptr,
                                c_ptr, c_i32, c_ptr, c_ptr, c_ptr]),
    "sa_shard_lengths": (c_i32, [c_ptr, c_i32, c_i32, c_i32, c_i32, c_ptr, c_ptr]),
    "sa_shard_selection": (c_i32, [c_ptr, c_ptr, c_i32, c_i32, c_i32, c_i32, c_ptr, c_ptr, c_i32, c_ptr,
                                   c_ptr]),
    "sa_merge_states": (c_i32, [c_ptr, c_ptr, c_i32, c_i32, c_i32, c_i32, c_ptr, c_ptr, c_ptr]),
    "sa_struct_size": (c_size, [c_i32]),
    "sa_wait_selftest": (c_i32, [c_i32, ctypes.c_int64, c_ptr, c_ptr, c_ptr]),
    "sa_status_string": (ctypes.c_char_p, [c_i32]),
    "sa_version": (ctypes.c_char_p, []),
}

_lib = None


def load():
    """Load the native library once (RuntimeError if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"native library {LIB_PATH} is missing: build it with "
            "`python -m sparse_paged_kv_page_gb300.build` (or __graft_entry__.build()); "
            "there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
