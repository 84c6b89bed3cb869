"""ctypes binding of libkvq.so (include/kvq.h).

Argument marshalling only: every step of the work runs in the CUDA kernels of
the shared library.  If the library has not been built, every entry point
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, byref, c_float, c_int32, c_int64, c_size_t, c_uint32, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

# kvq_status
KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_WORKSPACE = 3
KVQ_ERR_CUDA = 4

# bits of the device status word
KVQ_FLAG_SEQ_LEN = 0x1
KVQ_FLAG_BLOCK_TABLE = 0x2
KVQ_FLAG_ZERO_CLAMPED = 0x4
KVQ_FLAG_NONFINITE = 0x8
KVQ_FLAG_OOB = 0x10  # debug builds only: an access outside its array was skipped

# kvq_array: the caller arrays a debug build checks
(KVQ_ARRAY_K_CODES, KVQ_ARRAY_V_CODES, KVQ_ARRAY_K_SCALE, KVQ_ARRAY_K_ZERO, KVQ_ARRAY_V_SCALE,
 KVQ_ARRAY_V_ZERO, KVQ_ARRAY_K_WINDOW, KVQ_ARRAY_V_WINDOW, KVQ_ARRAY_BLOCK_TABLE, KVQ_ARRAY_Q,
 KVQ_ARRAY_K_NEW, KVQ_ARRAY_V_NEW, KVQ_ARRAY_SEQ_LENS, KVQ_ARRAY_OUT,
 KVQ_ARRAY_WORKSPACE) = range(15)

KVQ_DENSE = 0
KVQ_PAGED = 1


class kvq_cache_desc(Structure):
    _fields_ = [
        ("bits", c_int32),
        ("group_size", c_int32),
        ("num_kv_heads", c_int32),
        ("head_dim", c_int32),
        ("layout", c_int32),
        ("capacity", c_int32),
        ("num_pages", c_int32),
        ("max_blocks_per_seq", c_int32),
        ("symmetric", c_int32),
        ("k_per_channel", c_int32),
        ("sink_tokens", c_int32),
        ("nf4", c_int32),
    ]


class kvq_cache(Structure):
    _fields_ = [
        ("k_codes", c_void_p),
        ("v_codes", c_void_p),
        ("k_scale", c_void_p),
        ("k_zero", c_void_p),
        ("v_scale", c_void_p),
        ("v_zero", c_void_p),
        ("block_table", c_void_p),
        ("k_window", c_void_p),
        ("v_window", c_void_p),
    ]


class KVQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lib = None

# name -> (restype, argtypes): the C declarations of include/kvq.h
SIGNATURES = {
    "kvq_cache_bytes": (c_size_t, [POINTER(kvq_cache_desc), c_int64]),
    "kvq_cache_window_bytes": (c_size_t, [POINTER(kvq_cache_desc), c_int32]),
    "kvq_cache_array_bytes": (c_int32, [POINTER(kvq_cache_desc), c_int32,
                                        POINTER(c_size_t), POINTER(c_size_t)]),
    "kvq_append": (c_int32, [POINTER(kvq_cache_desc), POINTER(kvq_cache), c_int32, c_int32,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "kvq_decode_num_splits": (c_int32, [POINTER(kvq_cache_desc), c_int32, c_int32, c_int32,
                                        c_int32]),
    "kvq_decode_workspace_size": (c_size_t, [POINTER(kvq_cache_desc), c_int32, c_int32,
                                             c_int32, c_int32]),
    "kvq_decode_attn": (c_int32, [POINTER(kvq_cache_desc), POINTER(kvq_cache), c_int32, c_int32,
                                  c_void_p, c_void_p, c_int32, c_int32, c_float, c_void_p,
                                  c_void_p, c_size_t, c_void_p, c_void_p]),
    "kvq_append_decode_attn": (c_int32, [POINTER(kvq_cache_desc), POINTER(kvq_cache), c_int32,
                                         c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                         c_int32, c_float, c_void_p, c_void_p, c_size_t, c_void_p,
                                         c_void_p]),
    "kvq_decode_attn_static_ws": (c_int32, [POINTER(kvq_cache_desc), POINTER(kvq_cache), c_int32,
                                            c_int32, c_void_p, c_void_p, c_int32, c_int32,
                                            c_float, c_void_p, c_void_p, c_void_p]),
    "kvq_debug_checks": (c_int32, []),
    "kvq_debug_shrink_extent": (c_int32, [c_int32, c_int64]),
    "kvq_status_string": (ctypes.c_char_p, [c_int32]),
}


def load(path: str) -> ctypes.CDLL:
    """A handle on the library at `path` with the C signatures attached."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built; run `python -m quantized_kv_decode_gb300.build` "
            "(the library has no fallback path)")
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib() -> ctypes.CDLL:
    """Load libkvq.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def use(handle: ctypes.CDLL | None) -> ctypes.CDLL | None:
    """Route the binding's calls to `handle` (e.g. the debug build,
    libkvq_debug.so); None returns to libkvq.so.  Returns the previous handle."""
    global _lib
    prev, _lib = _lib, handle
    return prev


def status_string(status: int) -> str:
    return lib().kvq_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != KVQ_OK:
        raise KVQError(status, where)
