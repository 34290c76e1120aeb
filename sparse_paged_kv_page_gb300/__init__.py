"""GB300 (sm_103a) page-selected sparse decode over a paged KV cache.

The compute runs in the native library ``_sparse_attn.so`` (hand-written CUDA
for sm_103a behind the C ABI in include/sparse_attn.h); this package is its
thin torch binding plus the fused decode-step driver.
"""
from .api import *  # noqa: F401,F403
from .api import __all__ as _api_all

__all__ = list(_api_all)
