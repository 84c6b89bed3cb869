"""Seeded synthetic inputs for the tests and the benchmark.

This module holds no part of the method's arithmetic: it only draws random
K/V/q vectors, context lengths and block tables with the shapes of the
workloads below.  Both the CUDA path and the CPU oracle are fed from here.

Recipe (shared by every workload):
  * K and V entries ~ N(0, 1), drawn in fp32 and rounded to fp16.
  * K only: 4 channels per KV head, drawn once per cache with
    ``rng.choice(head_dim, 4, replace=False)`` and fixed for every token, are
    scaled by 10 (the persistent ~10x hot key channels of "What actually
    happens when you quantize a KV cache", section 3 step 7).
  * q ~ N(0, 1) in fp16.
  * Ragged lengths: ``rng.integers(lo, hi + 1)`` per sequence.
  * Paged caches: each sequence gets ceil(len / page_size) pages whose
    physical ids are consecutive runs of one ``rng.permutation`` of the
    pool; unused block-table entries are -1.
Host draws use numpy's PCG64 ``default_rng(seed)``; device draws (large
benchmark caches) use a seeded ``torch.Generator`` on the GPU.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    bits: tuple            # cache formats measured side by side (16 = fp16 cache)
    group_size: int
    ctx: tuple             # (lo, hi) cached tokens before the decode step
    layout: str = "dense"  # or "paged"
    page_size: int = 16
    layers: int = 1        # distinct per-layer caches one decode step walks
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def group_heads(self) -> int:
        return self.num_q_heads // self.num_kv_heads


# The five workloads of the build: shapes, formats and seeds.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 4, 128, (4,), 8, (256, 256), seed=0,
                     note="1 sequence, 4 heads, head_dim 128, context 256, INT4 group 8"),
    "mha7b": Workload("mha7b", 8, 32, 32, 128, (4, 16), 32, (4096, 4096), layers=32, seed=1,
                      note="7B-class MHA layer: batch 8 x 4096, 32 heads, INT4 g32 vs fp16"),
    "gqa_mix": Workload("gqa_mix", 64, 32, 8, 128, (4,), 64, (512, 8192), layers=32, seed=2,
                        note="GQA continuous-batching mix: batch 64, lengths U[512, 8192]"),
    "long": Workload("long", 4, 32, 8, 128, (8, 4), 32, (32768, 32768), layers=32, seed=3,
                     note="long context: batch 4 x 32768, INT8 and INT4 g32"),
    "paged": Workload("paged", 256, 14, 2, 64, (4,), 32, (128, 4096), layout="paged",
                      page_size=16, layers=24, seed=4,
                      note="paged 0.5B-class serving: batch 256, lengths U[128, 4096], 16-token pages"),
}


def rng_for(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def context_lengths(rng: np.random.Generator, batch: int, lo: int, hi: int) -> np.ndarray:
    if lo == hi:
        return np.full(batch, lo, dtype=np.int32)
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def outlier_channels(rng: np.random.Generator, num_kv_heads: int, head_dim: int,
                     count: int = 4) -> np.ndarray:
    return np.stack([rng.choice(head_dim, count, replace=False) for _ in range(num_kv_heads)])


def host_kv(rng: np.random.Generator, batch: int, tokens: int, num_kv_heads: int,
            head_dim: int, outliers: np.ndarray | None, outlier_gain: float = 10.0):
    """fp16 K and V [batch][tokens][kv_heads][head_dim]."""
    shape = (batch, tokens, num_kv_heads, head_dim)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    if outliers is not None:
        for h in range(num_kv_heads):
            k[:, :, h, outliers[h]] *= outlier_gain
    return k.astype(np.float16), v.astype(np.float16)


def host_q(rng: np.random.Generator, batch: int, num_q_heads: int, head_dim: int) -> np.ndarray:
    return rng.standard_normal((batch, num_q_heads, head_dim), dtype=np.float32).astype(np.float16)


def device_kv(gen, batch: int, tokens: int, num_kv_heads: int, head_dim: int,
              outliers: np.ndarray | None, device="cuda", outlier_gain: float = 10.0):
    """Like host_kv, drawn on the GPU from a seeded torch.Generator."""
    import torch
    shape = (batch, tokens, num_kv_heads, head_dim)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outliers is not None:
        for h in range(num_kv_heads):
            idx = torch.as_tensor(outliers[h], device=device, dtype=torch.long)
            k[:, :, h, idx] *= outlier_gain
    return k.half(), v.half()


def block_table(rng: np.random.Generator, lengths: np.ndarray, page_size: int,
                max_blocks: int | None = None, spare_pages: int = 0):
    """Scatter each sequence's pages over a pool by a seeded permutation.

    Returns (table int32 [batch][max_blocks], num_pages)."""
    need = [(int(n) + page_size - 1) // page_size for n in lengths]
    if max_blocks is None:
        max_blocks = max(1, max(need))
    num_pages = sum(need) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((len(lengths), max_blocks), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    return table, num_pages
