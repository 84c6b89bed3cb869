"""Test helpers: run one decode step through the C ABI and through the oracle
on the same seeded inputs.

The GPU side goes kvq_append (populate) -> kvq_append (one new token) ->
kvq_decode_attn.  The oracle side quantizes the same fp16 vectors with its
own quantizer and attends over its own dequantized cache.  Index work only
(gathering pages back into logical order) happens here.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle as O
from quantized_kv_decode_gb300 import synth

TOL_MAX_ABS = 2e-3   # max |gpu - oracle| over all outputs
TOL_REL_L2 = 1e-3    # ||gpu - oracle||_2 / ||oracle||_2


@dataclass
class Case:
    B: int
    Hq: int
    Hkv: int
    D: int
    bits: int
    g: int
    lens: np.ndarray          # cached tokens before the step
    layout: str = "dense"
    page_size: int = 16
    seed: int = 0
    spare_slots: int = 0      # extra dense capacity beyond max(lens)+1
    symmetric: bool = False   # absmax codes, scale only
    nf4: bool = False         # normal-quantile levels (bits 4), scale only


def make_inputs(c: Case):
    rng = synth.rng_for(c.seed)
    Lctx = int(max(c.lens.max(), 1))
    outl = synth.outlier_channels(rng, c.Hkv, c.D)
    k_ctx, v_ctx = synth.host_kv(rng, c.B, Lctx, c.Hkv, c.D, outl)
    k_new, v_new = synth.host_kv(rng, c.B, 1, c.Hkv, c.D, outl)
    q = synth.host_q(rng, c.B, c.Hq, c.D)
    table = num_pages = None
    if c.layout == "paged":
        # every sequence maps enough pages for the populate pass (Lctx) and the step
        need = np.full(c.B, Lctx + 1)
        table, num_pages = synth.block_table(rng, need, c.page_size, spare_pages=3)
    return dict(k_ctx=k_ctx, v_ctx=v_ctx, k_new=k_new, v_new=v_new, q=q, table=table,
                num_pages=num_pages, Lctx=Lctx)


def logical_rows(arr_np, c: Case, table, b, kvh, L):
    """Rows [0, L) of sequence b, KV head kvh, from a dense or paged array."""
    if c.layout == "dense":
        return arr_np[b, kvh, :L]
    pos = np.arange(L)
    pages = table[b, pos // c.page_size]
    return arr_np[pages, kvh, pos % c.page_size]


def run_gpu(c: Case, inp, num_splits=0, repeat=1, fused=False):
    """fused: the step's token is appended by kvq_append_decode_attn in the
    same call as the attention instead of a separate kvq_append."""
    import torch
    import quantized_kv_decode_gb300 as K
    dev = "cuda"
    Lctx = inp["Lctx"]
    cap = Lctx + 1 + c.spare_slots
    if c.layout == "dense":
        desc = K.make_desc(c.bits, c.g, c.Hkv, c.D, K.KVQ_DENSE, cap, symmetric=c.symmetric,
                           nf4=c.nf4)
        cache = K.KVCache.allocate(desc, c.B, dev)
    else:
        desc = K.make_desc(c.bits, c.g, c.Hkv, c.D, K.KVQ_PAGED, c.page_size,
                           inp["num_pages"], inp["table"].shape[1], symmetric=c.symmetric,
                           nf4=c.nf4)
        cache = K.KVCache.allocate(desc, c.B, dev, torch.from_numpy(inp["table"]))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    zeros = torch.zeros(c.B, dtype=torch.int32, device=dev)
    K.kvq_append(cache, torch.from_numpy(inp["k_ctx"]).to(dev), torch.from_numpy(inp["v_ctx"]).to(dev),
                 zeros, status)
    lens = torch.from_numpy(c.lens.astype(np.int32)).to(dev)
    k_new = torch.from_numpy(inp["k_new"]).to(dev)
    v_new = torch.from_numpy(inp["v_new"]).to(dev)
    if not fused:
        K.kvq_append(cache, k_new, v_new, lens, status)
    q = torch.from_numpy(inp["q"]).to(dev)
    outs = []
    for _ in range(repeat):
        if fused:
            o = K.kvq_append_decode_attn(cache, k_new[:, 0].contiguous(), v_new[:, 0].contiguous(),
                                         q, lens, Lctx + 1, dev_status=status,
                                         num_splits=num_splits)
        else:
            o = K.kvq_decode_attn(cache, q, lens + 1, Lctx + 1, dev_status=status,
                                  num_splits=num_splits)
        outs.append(o.cpu().numpy())
    torch.cuda.synchronize()
    return dict(out=outs[0], outs=outs, status=int(status.item()), cache=cache, desc=desc)


def oracle_step(c: Case, inp):
    """Oracle quantization of the logical cache and decode attention."""
    lens = c.lens.astype(np.int64)
    Lmax = int(lens.max()) + 1
    k_hat = np.zeros((c.B, c.Hkv, Lmax, c.D))
    v_hat = np.zeros((c.B, c.Hkv, Lmax, c.D))
    ref_codes = {}
    for which, ctx, new in (("k", inp["k_ctx"], inp["k_new"]), ("v", inp["v_ctx"], inp["v_new"])):
        hat = k_hat if which == "k" else v_hat
        for b in range(c.B):
            L = int(lens[b])
            rows = np.concatenate([ctx[b, :L], new[b, :1]], axis=0)   # [L+1][Hkv][D]
            rows = np.transpose(rows, (1, 0, 2))                        # [Hkv][L+1][D]
            if c.bits == 16:
                hat[b, :, :L + 1] = rows.astype(np.float64)
                ref_codes[(which, b)] = dict(raw=rows)
                continue
            if c.nf4:
                r = O.quantize_groups_nf4(rows, c.g)
                hat[b, :, :L + 1] = O.dequantize_nf4(r["codes"], r["scale"], c.g)
            else:
                quantize = O.quantize_groups_symmetric if c.symmetric else O.quantize_groups
                r = quantize(rows, c.bits, c.g)
                hat[b, :, :L + 1] = O.dequantize(r["codes"], r["scale"], r["zero"], c.g)
            ref_codes[(which, b)] = dict(packed=O.pack_codes(r["codes"], c.bits),
                                         scale=r["scale"], zero=r["zero"], flags=r["flags"])
    out = O.decode_attention(inp["q"], k_hat, v_hat, lens + 1)
    return out, ref_codes


def gpu_codes(run, c: Case, inp, which, b):
    """Logical (dequantization inputs) of sequence b from the GPU cache."""
    cache = run["cache"]
    L = int(c.lens[b]) + 1
    codes = (cache.k_codes if which == "k" else cache.v_codes).cpu().numpy()
    out = {}
    rows = [logical_rows(codes, c, inp["table"], b, h, L) for h in range(c.Hkv)]
    if c.bits == 16:
        out["raw"] = np.stack(rows).view(np.float16).reshape(c.Hkv, L, c.D)
        return out
    out["packed"] = np.stack(rows)
    for name in ("scale", "zero"):
        arr = getattr(cache, f"{which}_{name}")
        if arr is None:     # symmetric: the zero-point is the fixed code offset; NF4: none
            out[name] = None if c.nf4 else np.full_like(out["scale"], 1 << (c.bits - 1))
            continue
        t = arr.cpu().numpy()
        out[name] = np.stack([logical_rows(t, c, inp["table"], b, h, L) for h in range(c.Hkv)])
    return out


def assert_close(gpu, ref, tol_abs=TOL_MAX_ABS, tol_rel=TOL_REL_L2):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref)) / denom if denom > 0 else float(np.linalg.norm(gpu))
    assert max_abs <= tol_abs and rel <= tol_rel, f"max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel
