"""Full-size parity on sampled outputs.

Each workload runs at its full shape in the launch configuration the
benchmark uses (automatic split choice): caches populated by kvq_append from
seeded device-drawn fp16 K/V, then one kvq_append_decode_attn step (one new
token per sequence appended and attended in the same call).  For a few sampled (sequence, KV head) units the oracle
quantizes the same fp16 vectors (codes, scales and zeros must match
bit-exactly) and attends over them; the GPU output rows of that unit's query
heads must agree within the stated tolerance.
"""
import numpy as np
import pytest

import oracle as O
from quantized_kv_decode_gb300 import synth
from tests._cases import assert_close

pytestmark = pytest.mark.gpu


def _quantize(x, bits, g, kind):
    if kind == "sym":
        return O.quantize_groups_symmetric(x, bits, g)
    if kind == "nf4":
        return O.quantize_groups_nf4(x, g)
    return O.quantize_groups(x, bits, g)


def _dequantize(r, g, kind):
    if kind == "nf4":
        return O.dequantize_nf4(r["codes"], r["scale"], g)
    return O.dequantize(r["codes"], r["scale"], r["zero"], g)


def _run(w, bits, n_samples=3, seed_offset=0, kind="asym", group_size=None):
    import torch
    import quantized_kv_decode_gb300 as K
    dev = "cuda"
    rng = synth.rng_for(w.seed + seed_offset)
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    g = group_size or w.group_size
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
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    # populate: every sequence is written up to Lmax tokens; positions past a
    # paged sequence's own pages are flagged and skipped, so clear the word after
    K.kvq_append(cache, k_ctx, v_ctx, torch.zeros(B, dtype=torch.int32, device=dev), st)
    st.zero_()
    lens_t = torch.from_numpy(lens.astype(np.int32)).to(dev)
    # the step the benchmark times: one fused call
    out = K.kvq_append_decode_attn(cache, k_new[:, 0].contiguous(), v_new[:, 0].contiguous(), q,
                                   lens_t, Lmax + 1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    G = Hq // Hkv
    picks = [(0, 0), (B - 1, Hkv - 1)] + [(int(rng.integers(B)), int(rng.integers(Hkv)))
                                          for _ in range(max(0, n_samples - 2))]
    out_np = out.float().cpu().numpy()
    errs = []
    for b, kvh in picks:
        L = int(lens[b])
        kv_rows = []
        for which, ctx, new, codes_t in (("k", k_ctx, k_new, cache.k_codes),
                                         ("v", v_ctx, v_new, cache.v_codes)):
            x = torch.cat([ctx[b, :L, kvh], new[b, :1, kvh]]).cpu().numpy()   # [L+1][D] fp16
            pos = np.arange(L + 1)
            if w.layout == "dense":
                got_codes = codes_t[b, kvh, :L + 1].cpu().numpy()
                got_s = getattr(cache, f"{which}_scale")[b, kvh, :L + 1].cpu().numpy()
                zt = getattr(cache, f"{which}_zero")
                got_z = None if zt is None else zt[b, kvh, :L + 1].cpu().numpy()
            else:
                pages = torch.from_numpy(table_np[b, pos // w.page_size].astype(np.int64)).to(dev)
                offs = torch.from_numpy((pos % w.page_size).astype(np.int64)).to(dev)
                got_codes = codes_t[pages, kvh, offs].cpu().numpy()
                got_s = getattr(cache, f"{which}_scale")[pages, kvh, offs].cpu().numpy()
                zt = getattr(cache, f"{which}_zero")
                got_z = None if zt is None else zt[pages, kvh, offs].cpu().numpy()
            ref = _quantize(x, bits, g, kind)
            assert np.array_equal(got_codes, O.pack_codes(ref["codes"], bits)), (which, b, kvh)
            assert np.array_equal(got_s.view(np.uint16), ref["scale"].view(np.uint16))
            if got_z is not None:
                assert np.array_equal(got_z.view(np.uint16), ref["zero"].view(np.uint16))
            kv_rows.append(_dequantize(ref, g, kind))
        qh = q[b, kvh * G:(kvh + 1) * G].float().cpu().numpy().astype(np.float64)
        want = O.attend(qh, kv_rows[0], kv_rows[1], 1.0 / np.sqrt(D))
        errs.append(assert_close(out_np[b, kvh * G:(kvh + 1) * G], want))
    return errs


def test_fullsize_mha7b_int4():
    _run(synth.WORKLOADS["mha7b"], 4)


def test_fullsize_gqa_mix_int4():
    _run(synth.WORKLOADS["gqa_mix"], 4)


@pytest.mark.parametrize("bits", [8, 4])
def test_fullsize_long(bits):
    _run(synth.WORKLOADS["long"], bits, n_samples=2)


def test_fullsize_paged_int4():
    _run(synth.WORKLOADS["paged"], 4, n_samples=4)


@pytest.mark.parametrize("kind,bits,g", [("sym", 4, None), ("nf4", 4, 64), ("asym", 2, None),
                                         ("asym", 8, None)])
def test_fullsize_mha7b_formats(kind, bits, g):
    """The 7B-class workload in the benchmark's launch configuration for the
    comparator formats: symmetric INT4, NF4 g64, INT2, INT8."""
    _run(synth.WORKLOADS["mha7b"], bits, n_samples=2, kind=kind, group_size=g)
