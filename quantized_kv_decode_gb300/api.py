"""Python entry points over the C ABI, taking torch tensors.

PyTorch provides device memory and streams only.  Each function validates
dtypes and shapes, passes raw pointers to libkvq.so and returns; the kernels
do all the work.  Names follow include/kvq.h.
"""
from __future__ import annotations

import math
from ctypes import byref, c_size_t
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import (KVQ_DENSE, KVQ_PAGED, KVQError, kvq_cache, kvq_cache_desc)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def make_desc(bits: int, group_size: int, num_kv_heads: int, head_dim: int,
              layout: int = KVQ_DENSE, capacity: int = 0, num_pages: int = 0,
              max_blocks_per_seq: int = 0, symmetric: bool = False,
              k_per_channel: bool = False, sink_tokens: int = 0,
              nf4: bool = False) -> kvq_cache_desc:
    return kvq_cache_desc(bits, group_size, num_kv_heads, head_dim, layout, capacity,
                          num_pages, max_blocks_per_seq, int(bool(symmetric)),
                          int(bool(k_per_channel)), int(sink_tokens), int(bool(nf4)))


def kvq_cache_bytes(desc: kvq_cache_desc, tokens: int) -> int:
    return int(_lib.lib().kvq_cache_bytes(byref(desc), int(tokens)))


def kvq_cache_window_bytes(desc: kvq_cache_desc, batch: int) -> int:
    return int(_lib.lib().kvq_cache_window_bytes(byref(desc), int(batch)))


def kvq_cache_array_bytes(desc: kvq_cache_desc, batch: int) -> tuple[int, int]:
    cb, hb = c_size_t(0), c_size_t(0)
    _lib.check(_lib.lib().kvq_cache_array_bytes(byref(desc), int(batch), byref(cb), byref(hb)),
               "kvq_cache_array_bytes")
    return cb.value, hb.value


def kvq_decode_num_splits(desc, batch, num_q_heads, max_seq_len, num_splits=0) -> int:
    return int(_lib.lib().kvq_decode_num_splits(byref(desc), batch, num_q_heads, max_seq_len,
                                                num_splits))


def kvq_decode_workspace_size(desc, batch, num_q_heads, max_seq_len, num_splits=0) -> int:
    return int(_lib.lib().kvq_decode_workspace_size(byref(desc), batch, num_q_heads, max_seq_len,
                                                    num_splits))


def kvq_status_string(status: int) -> str:
    return _lib.status_string(status)


@dataclass
class KVCache:
    """One layer's quantized K/V cache: torch-owned device arrays + descriptor."""
    desc: kvq_cache_desc
    batch: int
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_scale: torch.Tensor | None
    k_zero: torch.Tensor | None
    v_scale: torch.Tensor | None
    v_zero: torch.Tensor | None
    block_table: torch.Tensor | None = None
    k_window: torch.Tensor | None = None
    v_window: torch.Tensor | None = None

    @classmethod
    def allocate(cls, desc: kvq_cache_desc, batch: int, device="cuda",
                 block_table: torch.Tensor | None = None) -> "KVCache":
        """Allocate zeroed arrays in the layout include/kvq.h documents."""
        D, Hkv = desc.head_dim, desc.num_kv_heads
        row_bytes = D * desc.bits // 8
        if desc.layout == KVQ_DENSE:
            lead = (batch, Hkv, desc.capacity)
        else:
            lead = (desc.num_pages, Hkv, desc.capacity)
            if block_table is None:
                raise ValueError("a paged cache needs a block table")
            block_table = block_table.to(device=device, dtype=torch.int32).contiguous()
        codes = lambda: torch.zeros(lead + (row_bytes,), dtype=torch.uint8, device=device)
        if desc.bits == 16:
            hdr = lambda: None
        else:
            ng = D // desc.group_size
            hdr = lambda: torch.zeros(lead + (ng,), dtype=torch.float16, device=device)
        zero = (lambda: None) if (desc.symmetric or desc.nf4) else hdr
        if desc.k_per_channel:
            # K: one scale + zero per channel for each block of g tokens
            g = desc.group_size
            # (paged: per page; the pages hold the tokens after the sinks)
            khdr = lambda: torch.zeros((lead[0], Hkv, desc.capacity // g, D), dtype=torch.float16,
                                       device=device)
            win = lambda: torch.zeros((batch, Hkv, desc.sink_tokens + g, D), dtype=torch.float16,
                                      device=device)
            return cls(desc, batch, codes(), codes(), khdr(), khdr(), hdr(), hdr(), block_table,
                       win(), win())
        return cls(desc, batch, codes(), codes(), hdr(), zero(), hdr(), zero(), block_table)

    @property
    def ptrs(self) -> kvq_cache:
        return kvq_cache(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_scale),
                         _ptr(self.k_zero), _ptr(self.v_scale), _ptr(self.v_zero),
                         _ptr(self.block_table), _ptr(self.k_window), _ptr(self.v_window))

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.k_codes, self.v_codes, self.k_scale, self.k_zero, self.v_scale,
                    self.v_zero, self.k_window, self.v_window) if t is not None)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor of dtype {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def kvq_append(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor,
               seq_lens_before: torch.Tensor, dev_status: torch.Tensor | None = None,
               stream=None) -> None:
    """Quantize k_new/v_new [B][T][Hkv][D] fp16 into the cache at positions
    seq_lens_before[b] + t."""
    _need(k_new, torch.float16, "k_new", 4)
    _need(v_new, torch.float16, "v_new", 4)
    _need(seq_lens_before, torch.int32, "seq_lens_before", 1)
    if k_new.shape != v_new.shape:
        raise ValueError("k_new and v_new must have the same shape")
    B, T, Hkv, D = k_new.shape
    if Hkv != cache.desc.num_kv_heads or D != cache.desc.head_dim or seq_lens_before.numel() != B:
        raise ValueError("shape does not match the cache descriptor")
    st = _lib.lib().kvq_append(byref(cache.desc), byref(cache.ptrs), B, T, _ptr(k_new),
                               _ptr(v_new), _ptr(seq_lens_before), _ptr(dev_status),
                               _stream(stream))
    _lib.check(st, "kvq_append")


def kvq_decode_attn(cache: KVCache, q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    dev_status: torch.Tensor | None = None, num_splits: int = 0,
                    softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
    """Decode attention of q [B][Hq][D] fp16 over the cache; returns out."""
    _need(q, torch.float16, "q", 3)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, Hq, D = q.shape
    if D != cache.desc.head_dim or seq_lens.numel() != B:
        raise ValueError("shape does not match the cache descriptor")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float16, "out", 3)
    need = kvq_decode_workspace_size(cache.desc, B, Hq, max_seq_len, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.lib().kvq_decode_attn(byref(cache.desc), byref(cache.ptrs), B, Hq, _ptr(q),
                                    _ptr(seq_lens), int(max_seq_len), int(num_splits),
                                    float(softmax_scale), _ptr(out), _ptr(workspace), ws_bytes,
                                    _ptr(dev_status), _stream(stream))
    _lib.check(st, "kvq_decode_attn")
    return out


def kvq_append_decode_attn(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                           q: torch.Tensor, seq_lens_before: torch.Tensor, max_seq_len: int,
                           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           dev_status: torch.Tensor | None = None, num_splits: int = 0,
                           softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
    """One decode step: append k_new/v_new [B][Hkv][D] at seq_lens_before and
    attend q [B][Hq][D] over seq_lens_before + 1 tokens; returns out."""
    _need(q, torch.float16, "q", 3)
    _need(k_new, torch.float16, "k_new", 3)
    _need(v_new, torch.float16, "v_new", 3)
    _need(seq_lens_before, torch.int32, "seq_lens_before", 1)
    B, Hq, D = q.shape
    if (D != cache.desc.head_dim or seq_lens_before.numel() != B
            or tuple(k_new.shape) != (B, cache.desc.num_kv_heads, D)
            or tuple(v_new.shape) != tuple(k_new.shape)):
        raise ValueError("shape does not match the cache descriptor")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float16, "out", 3)
    need = kvq_decode_workspace_size(cache.desc, B, Hq, max_seq_len, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.lib().kvq_append_decode_attn(
        byref(cache.desc), byref(cache.ptrs), B, Hq, _ptr(k_new), _ptr(v_new), _ptr(q),
        _ptr(seq_lens_before), int(max_seq_len), int(num_splits), float(softmax_scale), _ptr(out),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _lib.check(st, "kvq_append_decode_attn")
    return out


def kvq_decode_attn_static_ws(cache: KVCache, q: torch.Tensor, seq_lens: torch.Tensor,
                              max_seq_len: int, out: torch.Tensor,
                              dev_status: torch.Tensor | None = None, num_splits: int = 0,
                              softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
    """kvq_decode_attn with the library's static split scratch instead of a
    workspace; allocates nothing, so `out` must be given.  Calls that can
    overlap on the GPU share that scratch and race."""
    _need(q, torch.float16, "q", 3)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(out, torch.float16, "out", 3)
    B, Hq, D = q.shape
    if D != cache.desc.head_dim or seq_lens.numel() != B or out.shape != q.shape:
        raise ValueError("shape does not match the cache descriptor")
    st = _lib.lib().kvq_decode_attn_static_ws(
        byref(cache.desc), byref(cache.ptrs), B, Hq, _ptr(q), _ptr(seq_lens), int(max_seq_len),
        int(num_splits), float(softmax_scale), _ptr(out), _ptr(dev_status), _stream(stream))
    _lib.check(st, "kvq_decode_attn_static_ws")
    return out


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
