"""Full-size parity.

Each workload runs at its full shape in the launch configuration the
benchmark uses (automatic split choice): caches populated by kvq_append from
seeded device-drawn fp16 K/V, then one kvq_append_decode_attn step (one new
token per sequence appended and attended in the same call).  The 7B-class
INT4 step and the paged small-model step are checked on every (sequence, KV
head) unit; the other workloads and formats on sampled units.  For each
checked unit the oracle quantizes the same fp16 vectors (codes, scales and
zeros must match bit-exactly) and attends over them; the GPU output rows of
that unit's query heads must agree within the stated tolerance.  Every cache
array and the output sit between guard bytes that must be intact after the
step.
"""
import os

import numpy as np
import pytest

from quantized_kv_decode_gb300 import synth
from tests._cases import Guarded, check_guards, check_units, guarded_cache

pytestmark = pytest.mark.gpu


def _run(w, bits, n_samples=3, seed_offset=0, kind="asym", group_size=None):
    """n_samples: units to check, or None for every (sequence, KV head) unit."""
    import torch
    import quantized_kv_decode_gb300 as K
    dev = "cuda"
    rng = synth.rng_for(w.seed + seed_offset)
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    g = w.group_size if group_size is None else group_size
    opts = dict(symmetric=kind == "sym", nf4=kind == "nf4")
    lens = synth.context_lengths(rng, B, *w.ctx)            # cached tokens before the step
    Lmax = int(lens.max())
    outl = synth.outlier_channels(rng, Hkv, D)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 7919 + seed_offset)
    k_ctx, v_ctx = synth.device_kv(gen, B, Lmax, Hkv, D, outl, dev)
    k_new, v_new = synth.device_kv(gen, B, 1, Hkv, D, outl, dev)
    q = torch.randn((B, Hq, D), generator=gen, device=dev).half()

    table_np = None
    if w.layout == "dense":
        desc = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, ((Lmax + 1 + 15) // 16) * 16, **opts)
        cache = K.KVCache.allocate(desc, B, dev)
    else:
        # each sequence owns ceil((len + 1) / page_size) pages, scattered over the pool
        table_np, num_pages = synth.block_table(rng, lens + 1, w.page_size)
        desc = K.make_desc(bits, g, Hkv, D, K.KVQ_PAGED, w.page_size, num_pages, table_np.shape[1],
                           **opts)
        cache = K.KVCache.allocate(desc, B, dev, torch.from_numpy(table_np))
    cache, guards = guarded_cache(cache)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    # populate: every sequence is written up to Lmax tokens; positions past a
    # paged sequence's own pages are flagged and skipped, so clear the word after
    K.kvq_append(cache, k_ctx, v_ctx, torch.zeros(B, dtype=torch.int32, device=dev), st)
    st.zero_()
    lens_t = torch.from_numpy(lens.astype(np.int32)).to(dev)
    # the step the benchmark times: one fused call
    guards["out"] = Guarded(q.shape, torch.float16, dev)
    ws_bytes = K.kvq_decode_workspace_size(desc, B, Hq, Lmax + 1, 0)
    if ws_bytes:
        guards["workspace"] = Guarded((ws_bytes,), torch.uint8, dev)
    out = K.kvq_append_decode_attn(cache, k_new[:, 0].contiguous(), v_new[:, 0].contiguous(), q,
                                   lens_t, Lmax + 1, out=guards["out"].tensor,
                                   workspace=guards["workspace"].tensor if ws_bytes else None,
                                   dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_guards(guards, "fused step")

    G = Hq // Hkv
    if n_samples is None:
        picks = {b: list(range(Hkv)) for b in range(B)}
    else:
        picks = {}
        for b, kvh in [(0, 0), (B - 1, Hkv - 1)] + [(int(rng.integers(B)), int(rng.integers(Hkv)))
                                                    for _ in range(max(0, n_samples - 2))]:
            picks.setdefault(b, [])
            if kvh not in picks[b]:
                picks[b].append(kvh)
    out_np = out.float().cpu().numpy()
    q_np = q.float().cpu().numpy()
    jobs = []
    for b, heads in sorted(picks.items()):
        # the picked KV heads of sequence b at once: [heads][L+1][D]
        L = int(lens[b])
        hs = torch.tensor(heads, device=dev)
        pos = np.arange(L + 1)
        x, got = {}, {}
        for which, ctx, new, codes_t in (("k", k_ctx, k_new, cache.k_codes),
                                         ("v", v_ctx, v_new, cache.v_codes)):
            x[which] = torch.cat([ctx[b, :L], new[b, :1]])[:, hs].transpose(0, 1).cpu().numpy()
            arrays = [codes_t, getattr(cache, f"{which}_scale"), getattr(cache, f"{which}_zero")]
            if w.layout == "dense":
                got[which] = tuple(None if t is None else t[b, hs, :L + 1].cpu().numpy()
                                   for t in arrays)
            else:
                pages = torch.from_numpy(table_np[b, pos // w.page_size].astype(np.int64)).to(dev)
                offs = torch.from_numpy((pos % w.page_size).astype(np.int64)).to(dev)
                got[which] = tuple(
                    None if t is None else t[pages[None, :], hs[:, None], offs[None, :]].cpu().numpy()
                    for t in arrays)
        qh = np.stack([q_np[b, kvh * G:(kvh + 1) * G] for kvh in heads])
        oh = np.stack([out_np[b, kvh * G:(kvh + 1) * G] for kvh in heads])
        jobs.append((x["k"], x["v"], got, qh, oh, bits, g, kind, (b, heads)))
    if len(jobs) == 1:
        return check_units(jobs[0])
    # the oracle is plain fp64 numpy: spread the sequences over host cores
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    workers = max(1, min(len(jobs), 8, os.cpu_count() or 1))
    errs = []
    with ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        for r in ex.map(check_units, jobs):
            errs.extend(r)
    return errs


def test_fullsize_mha7b_int4():
    """Every (sequence, KV head) unit of the 7B-class step."""
    _run(synth.WORKLOADS["mha7b"], 4, n_samples=None)


def test_fullsize_gqa_mix_int4():
    _run(synth.WORKLOADS["gqa_mix"], 4, n_samples=16)


@pytest.mark.parametrize("bits", [8, 4])
def test_fullsize_long(bits):
    _run(synth.WORKLOADS["long"], bits, n_samples=6)


def test_fullsize_paged_int4():
    """Every (sequence, KV head) unit of the paged small-model step."""
    _run(synth.WORKLOADS["paged"], 4, n_samples=None)


@pytest.mark.parametrize("kind,bits,g", [("sym", 4, None), ("nf4", 4, 64), ("asym", 2, None),
                                         ("asym", 8, None), ("fp16", 16, 0)])
def test_fullsize_mha7b_formats(kind, bits, g):
    """The 7B-class workload in the benchmark's launch configuration for the
    comparator formats: symmetric INT4, NF4 g64, INT2, INT8, and the fp16
    cache (the tensor-core fp16 kernel)."""
    _run(synth.WORKLOADS["mha7b"], bits, n_samples=8, kind=kind, group_size=g)
