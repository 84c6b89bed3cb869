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


class Guarded:
    """A device tensor housed inside a larger byte buffer whose PAD bytes on
    either side (and any tail bytes up to the next 16) hold PATTERN, so that a
    kernel writing outside the tensor is caught by intact()."""
    PAD = 4096
    PATTERN = 0xA5

    def __init__(self, shape, dtype, device):
        import torch
        n = 1
        for d in shape:
            n *= int(d)
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        span = (self.nbytes + 15) // 16 * 16
        self.buf = torch.full((2 * self.PAD + span,), self.PATTERN, dtype=torch.uint8,
                              device=device)
        self.tensor = self.buf[self.PAD:self.PAD + self.nbytes].view(dtype).view(tuple(shape))
        self.tensor.zero_()

    def intact(self) -> bool:
        return bool((self.buf[:self.PAD] == self.PATTERN).all()) and bool(
            (self.buf[self.PAD + self.nbytes:] == self.PATTERN).all())


CACHE_ARRAYS = ("k_codes", "v_codes", "k_scale", "k_zero", "v_scale", "v_zero", "k_window",
                "v_window")


def guarded_cache(cache):
    """The same cache (descriptor, shapes, zeroed contents, block table) with
    every array moved into a Guarded buffer; returns (cache, guards)."""
    import quantized_kv_decode_gb300 as K
    guards, arrays = {}, {}
    for name in CACHE_ARRAYS:
        t = getattr(cache, name)
        if t is None:
            arrays[name] = None
            continue
        g = Guarded(t.shape, t.dtype, t.device)
        guards[name] = g
        arrays[name] = g.tensor
    return K.KVCache(cache.desc, cache.batch, block_table=cache.block_table, **arrays), guards


def check_guards(guards: dict, where: str):
    bad = [name for name, g in guards.items() if not g.intact()]
    assert not bad, f"{where}: bytes written outside {bad}"


def run_gpu(c: Case, inp, num_splits=0, repeat=1, fused=False, ws_fill=None):
    """ws_fill: a byte written over the whole split workspace before the calls
    (its contents need no init).  fused: the step's token is appended by kvq_append_decode_attn in the
    same call as the attention instead of a separate kvq_append.  Every cache
    array, the output and the split workspace sit between guard bytes that
    are checked after each call."""
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
    cache, guards = guarded_cache(cache)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    zeros = torch.zeros(c.B, dtype=torch.int32, device=dev)
    K.kvq_append(cache, torch.from_numpy(inp["k_ctx"]).to(dev), torch.from_numpy(inp["v_ctx"]).to(dev),
                 zeros, status)
    check_guards(guards, "populate")
    lens = torch.from_numpy(c.lens.astype(np.int32)).to(dev)
    k_new = torch.from_numpy(inp["k_new"]).to(dev)
    v_new = torch.from_numpy(inp["v_new"]).to(dev)
    if not fused:
        K.kvq_append(cache, k_new, v_new, lens, status)
        check_guards(guards, "append")
    q = torch.from_numpy(inp["q"]).to(dev)
    ws_bytes = K.kvq_decode_workspace_size(desc, c.B, c.Hq, Lctx + 1, num_splits)
    if ws_bytes:
        guards["workspace"] = Guarded((ws_bytes,), torch.uint8, dev)
    ws = guards["workspace"].tensor if ws_bytes else None
    if ws is not None and ws_fill is not None:
        ws.fill_(ws_fill)
    outs = []
    for _ in range(repeat):
        guards["out"] = Guarded(q.shape, torch.float16, dev)
        o = guards["out"].tensor
        if fused:
            K.kvq_append_decode_attn(cache, k_new[:, 0].contiguous(), v_new[:, 0].contiguous(),
                                     q, lens, Lctx + 1, out=o, workspace=ws, dev_status=status,
                                     num_splits=num_splits)
        else:
            K.kvq_decode_attn(cache, q, lens + 1, Lctx + 1, out=o, workspace=ws,
                              dev_status=status, num_splits=num_splits)
        check_guards(guards, "fused step" if fused else "decode")
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


def _quantize_any(x, bits, g, kind):
    if kind == "sym":
        return O.quantize_groups_symmetric(x, bits, g)
    if kind == "nf4":
        return O.quantize_groups_nf4(x, g)
    return O.quantize_groups(x, bits, g)


def _dequantize_any(r, g, kind):
    if kind == "nf4":
        return O.dequantize_nf4(r["codes"], r["scale"], g)
    return O.dequantize(r["codes"], r["scale"], r["zero"], g)


def check_units(job):
    """Oracle check of some KV heads of one sequence (a process-pool job).

    job: x_k, x_v fp16 [heads][L][D] (the rows the GPU quantized, the new one
    last); got: {"k"/"v": (packed codes, scale, zero or None)} read back from
    the GPU cache for those rows; q [heads][G][D]; out [heads][G][D] the
    GPU's fp16 output rows; bits, g, kind.  Codes, scales and zeros must be
    bit-identical to the oracle's; the output within the decode tolerance.
    Returns (max_abs, rel_l2) per head."""
    x_k, x_v, got, q, out, bits, g, kind, tag = job
    hats = []
    for which, x in (("k", x_k), ("v", x_v)):
        if bits == 16:  # fp16 cache: the append copies the rows
            codes = got[which][0]
            assert np.array_equal(codes.view(np.uint16).reshape(x.shape), x.view(np.uint16)), (tag, which)
            hats.append(x.astype(np.float64))
            continue
        ref = _quantize_any(x, bits, g, kind)
        codes, scale, zero = got[which]
        assert np.array_equal(codes, O.pack_codes(ref["codes"], bits)), (tag, which, "codes")
        assert np.array_equal(scale.view(np.uint16), ref["scale"].view(np.uint16)), (tag, which)
        if zero is not None:
            assert np.array_equal(zero.view(np.uint16), ref["zero"].view(np.uint16)), (tag, which)
        hats.append(_dequantize_any(ref, g, kind))
    D = x_k.shape[-1]
    return [assert_close(out[i], O.attend(q[i].astype(np.float64), hats[0][i], hats[1][i],
                                          1.0 / np.sqrt(D)))
            for i in range(x_k.shape[0])]
