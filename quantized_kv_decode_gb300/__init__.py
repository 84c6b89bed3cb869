"""Quantized KV-cache decode attention for GB300 (sm_103a).

The work runs in libkvq.so (CUDA kernels behind the C ABI of include/kvq.h);
this package is its thin Python binding plus a seeded synthetic-input module.
Build the library with ``python -m quantized_kv_decode_gb300.build``.
"""
from ._lib import (KVQ_DENSE, KVQ_ERR_CUDA, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED,  # noqa: F401
                   KVQ_ERR_WORKSPACE, KVQ_FLAG_BLOCK_TABLE, KVQ_FLAG_NONFINITE, KVQ_FLAG_OOB,
                   KVQ_FLAG_SEQ_LEN, KVQ_FLAG_ZERO_CLAMPED, KVQ_OK, KVQ_PAGED, KVQError,
                   kvq_cache, kvq_cache_desc, lib)

__all__ = [
    "KVCache", "make_desc", "kvq_append", "kvq_decode_attn", "kvq_append_decode_attn",
    "kvq_decode_attn_static_ws", "kvq_cache_bytes",
    "kvq_cache_array_bytes", "kvq_cache_window_bytes", "kvq_decode_num_splits", "kvq_decode_workspace_size",
    "kvq_status_string", "KVQError", "lib",
]


def __getattr__(name):
    # the torch-facing API is imported lazily so that the input generators and
    # the ctypes layer can be used without importing torch
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
