"""GB300-native GraniKV decode-step attention over an asymmetric HOT/COLD KV cache.

GraniKV (arXiv:2608.15584) keeps each long shared prefix in a contiguous HOT slab and each
request's suffix and decoded tokens in a token-level COLD pool, and picks per decode step
between a dense batched-GEMM prefix backend and a cascade backend that reads the prefix once.

The work runs in ``libgranikv.so`` (C ABI in include/granikv.h, CUDA kernels for sm_103a);
this package is its thin binding.  Build the library with
``python -m shared_prefix_kv_decode_gb300.build``; without it every call raises.
"""

from ._binding import (  # noqa: F401
    BACKEND_AUTO, BACKEND_CASCADE, BACKEND_DENSE, BACKEND_NAMES, DTYPE_BF16, DTYPE_F32,
    Batch, Context, DeviceCheckFailed, GranikvError, NoColdSpace, NoHotSpace, Plan,
    load_library, status_string,
)

__all__ = [
    "BACKEND_AUTO", "BACKEND_CASCADE", "BACKEND_DENSE", "BACKEND_NAMES", "DTYPE_BF16", "DTYPE_F32",
    "Batch", "Context", "DeviceCheckFailed", "GranikvError", "NoColdSpace", "NoHotSpace", "Plan",
    "load_library", "status_string", "GraniKVCache",
]


def __getattr__(name):
    if name == "GraniKVCache":
        from .cache import GraniKVCache
        return GraniKVCache
    raise AttributeError(name)
