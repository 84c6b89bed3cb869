"""GPU parity of axis-aware (KIVI-style) caches against the oracle.

K is grouped per channel over blocks of g tokens, V per token; the first
sink tokens and the newest tokens that have not filled a block stay fp16.
Caches are filled by kvq_append calls of several sizes (one token at a time,
uneven chunks, everything at once); the stored codes, per-channel K headers,
per-token V headers and fp16 window must equal oracle.kivi_quantize bit for
bit, and kvq_decode_attn / kvq_append_decode_attn must match the oracle's
attention over the dequantized cache within the decode tolerance (max |err|
<= 2e-3, relative L2 <= 1e-3).
"""
import numpy as np
import pytest

import oracle as O
from quantized_kv_decode_gb300 import synth
from tests._cases import assert_close

pytestmark = pytest.mark.gpu


def _seq_view(K, cache, b):
    """A one-sequence view of a dense cache (slices of the batch arrays)."""
    sl = slice(b, b + 1)
    return K.KVCache(cache.desc, 1, cache.k_codes[sl], cache.v_codes[sl], cache.k_scale[sl],
                     cache.k_zero[sl], cache.v_scale[sl], cache.v_zero[sl], None,
                     cache.k_window[sl], cache.v_window[sl])


def _paged_view(K, cache, b):
    """A one-sequence view of a paged cache: the shared page pool, row b of
    the block table and of the fp16 window."""
    sl = slice(b, b + 1)
    return K.KVCache(cache.desc, 1, cache.k_codes, cache.v_codes, cache.k_scale, cache.k_zero,
                     cache.v_scale, cache.v_zero, cache.block_table[sl], cache.k_window[sl],
                     cache.v_window[sl])


def _fill(K, cache, k, v, lens, chunks, st, view_fn=None):
    """Append sequence b's first lens[b] tokens in pieces of the given sizes."""
    import torch
    for b, L in enumerate(lens):
        view = (view_fn or _seq_view)(K, cache, b)
        pos, i = 0, 0
        while pos < L:
            n = min(chunks[i % len(chunks)], L - pos)
            K.kvq_append(view, k[b:b + 1, pos:pos + n].contiguous(), v[b:b + 1, pos:pos + n].contiguous(),
                         torch.tensor([pos], dtype=torch.int32, device="cuda"), st)
            pos += n
            i += 1


def _compare_cache(cache, k16, v16, lens, bits, g, S):
    """Stored parts against the oracle, per sequence."""
    for b, L in enumerate(lens):
        kk = np.transpose(k16[b, :L], (1, 0, 2))           # [Hkv][L][D]
        vv = np.transpose(v16[b, :L], (1, 0, 2))
        r = O.kivi_quantize(kk, vv, bits, g, S)
        S_, nb, r0 = r["S"], r["nb"], r["r0"]
        kc = cache.k_codes[b].cpu().numpy()
        vc = cache.v_codes[b].cpu().numpy()
        assert np.array_equal(kc[:, S_:r0], O.pack_codes(r["k_codes"], bits)), b
        assert np.array_equal(vc[:, S_:r0], O.pack_codes(r["v_codes"], bits)), b
        for name, want in (("k_scale", r["k_scale"]), ("k_zero", r["k_zero"])):
            got = getattr(cache, name)[b, :, :nb].cpu().numpy()
            assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), (name, b)
        for name, want in (("v_scale", r["v_scale"]), ("v_zero", r["v_zero"])):
            got = getattr(cache, name)[b, :, S_:r0].cpu().numpy()
            assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), (name, b)
        kw = cache.k_window[b].cpu().numpy()
        vw = cache.v_window[b].cpu().numpy()
        assert np.array_equal(kw[:, :S_].view(np.uint16), kk[:, :S_].view(np.uint16))
        assert np.array_equal(vw[:, :S_].view(np.uint16), vv[:, :S_].view(np.uint16))
        for p in range(r0, L):
            slot = S + (p - S) % g
            assert np.array_equal(kw[:, slot].view(np.uint16), kk[:, p].view(np.uint16)), (b, p)
            assert np.array_equal(vw[:, slot].view(np.uint16), vv[:, p].view(np.uint16)), (b, p)


def _oracle_out(q16, k16, v16, lens, bits, g, S):
    B, Hq, D = q16.shape
    Hkv = k16.shape[2]
    Lmax = int(max(lens))
    k_hat = np.zeros((B, Hkv, Lmax, D))
    v_hat = np.zeros((B, Hkv, Lmax, D))
    for b, L in enumerate(lens):
        r = O.kivi_quantize(np.transpose(k16[b, :L], (1, 0, 2)), np.transpose(v16[b, :L], (1, 0, 2)),
                            bits, g, S)
        k_hat[b, :, :L] = r["k_hat"]
        v_hat[b, :, :L] = r["v_hat"]
    return O.decode_attention(q16, k_hat, v_hat, np.asarray(lens))


def _run(bits, g, S, D, Hq, Hkv, lens, chunks, splits=0, seed=0, cap=None):
    import torch
    import quantized_kv_decode_gb300 as K
    B = len(lens)
    Lmax = int(max(lens))
    cap = cap or ((Lmax + 1 + g - 1) // g) * g + g
    rng = synth.rng_for(seed)
    outl = synth.outlier_channels(rng, Hkv, D)
    k16, v16 = synth.host_kv(rng, B, Lmax + 1, Hkv, D, outl)
    q16 = synth.host_q(rng, B, Hq, D)
    desc = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, cap, k_per_channel=True, sink_tokens=S)
    cache = K.KVCache.allocate(desc, B)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kt, vt = torch.from_numpy(k16).cuda(), torch.from_numpy(v16).cuda()
    _fill(K, cache, kt, vt, lens, chunks, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare_cache(cache, k16, v16, lens, bits, g, S)
    q = torch.from_numpy(q16).cuda()
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = K.kvq_decode_attn(cache, q, lt, Lmax, dev_status=st, num_splits=splits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out.cpu().numpy(), _oracle_out(q16, k16, v16, lens, bits, g, S))
    return K, cache, k16, v16, q16, kt, vt, q, lt, st


@pytest.mark.parametrize("bits,g,S,D,Hq,Hkv", [
    (4, 32, 4, 128, 8, 2), (8, 32, 0, 128, 4, 4), (4, 64, 16, 128, 4, 1), (4, 16, 1, 64, 14, 2),
    (8, 128, 8, 128, 2, 2), (4, 32, 3, 256, 4, 2)])
def test_kivi_append_bit_exact_and_decode(bits, g, S, D, Hq, Hkv):
    lens = [0, 1, S, S + g - 1, S + g, S + 3 * g + 5, 300]
    lens = [L for L in lens if L > 0]
    _run(bits, g, S, D, Hq, Hkv, lens, chunks=[1, 7, 64, 3], seed=bits + g + S + D)


@pytest.mark.parametrize("bits,g,S,D,Hq,Hkv", [
    (4, 32, 4, 128, 32, 32), (4, 64, 2, 128, 8, 2), (8, 32, 0, 128, 16, 2), (4, 32, 8, 64, 14, 2)])
@pytest.mark.parametrize("splits", [0, 5])
def test_kivi_long_contexts(bits, g, S, D, Hq, Hkv, splits):
    """Thousands of tokens: many blocks per warp, several splits, a residual
    window of every fill (the tensor-core path for g a multiple of 32)."""
    lens = [S + 40 * g + 17, 2051, S + 3 * g]
    _run(bits, g, S, D, Hq, Hkv, lens, chunks=[2048, 1, 300], splits=splits, seed=bits * g + S)


@pytest.mark.parametrize("chunks", [[1], [1000], [5, 11, 2]])
def test_kivi_append_granularity_does_not_matter(chunks):
    """The same tokens appended one at a time, all at once, or in uneven
    pieces give the same cache (checked bit-exact against the oracle)."""
    _run(4, 32, 4, 128, 8, 2, [173, 64, 37], chunks=chunks, seed=77)


@pytest.mark.parametrize("splits", [1, 3])
def test_kivi_fused_step_and_splits(splits):
    """kvq_append_decode_attn on an axis-aware cache: the step's token lands
    in the residual window (or completes a block) and is attended."""
    import torch
    g, S = 32, 4
    lens = [S + 2 * g - 1, S + 5, 150]          # the first sequence completes a block
    K, cache, k16, v16, q16, kt, vt, q, lt, st = _run(4, g, S, 128, 8, 2, lens, [16],
                                                      splits=splits, seed=5)
    new_k = torch.stack([kt[b, L] for b, L in enumerate(lens)]).contiguous()   # [B][Hkv][D]
    new_v = torch.stack([vt[b, L] for b, L in enumerate(lens)]).contiguous()
    out = K.kvq_append_decode_attn(cache, new_k, new_v, q, lt, max(lens) + 1, dev_status=st,
                                   num_splits=splits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lens1 = [L + 1 for L in lens]
    _compare_cache(cache, k16, v16, lens1, 4, g, S)
    assert_close(out.cpu().numpy(), _oracle_out(q16, k16, v16, lens1, 4, g, S))


def test_kivi_descriptor_limits():
    import torch
    import quantized_kv_decode_gb300 as K
    # paged: a page must hold whole blocks
    paged = K.make_desc(4, 32, 2, 128, K.KVQ_PAGED, 48, 10, 4, k_per_channel=True)
    with pytest.raises(K.KVQError) as e:
        K.kvq_cache_array_bytes(paged, 1)
    assert e.value.status == K.KVQ_ERR_INVALID_ARG
    # appending past the capacity flags SEQ_LEN and writes nothing there
    desc = K.make_desc(4, 32, 2, 128, K.KVQ_DENSE, 64, k_per_channel=True, sink_tokens=4)
    cache = K.KVCache.allocate(desc, 1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3)
    x = torch.randn((1, 70, 2, 128), generator=gen, device="cuda").half()
    y = torch.randn((1, 70, 2, 128), generator=gen, device="cuda").half()
    K.kvq_append(cache, x, y, torch.zeros(1, dtype=torch.int32, device="cuda"), st)
    torch.cuda.synchronize()
    assert int(st.item()) == K.KVQ_FLAG_SEQ_LEN
    # the 64 positions inside the cache hold the first 64 tokens
    k16, v16 = x.cpu().numpy(), y.cpu().numpy()
    _compare_cache(cache, k16, v16, [64], 4, 32, 4)
    q16 = torch.randn((1, 4, 128), generator=gen, device="cuda").half()
    st.zero_()
    out = K.kvq_decode_attn(cache, q16, torch.tensor([64], dtype=torch.int32, device="cuda"), 64,
                            dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out.cpu().numpy(), _oracle_out(q16.cpu().numpy(), k16, v16, [64], 4, 32, 4))


def test_kivi_fullsize_mha7b():
    """The 7B-class workload (batch 8 x 4096 cached tokens, 32 heads, head_dim
    128, INT4 g32, 4 sinks) in the benchmark's configuration: one populating
    append, one fused step; sampled units checked against the oracle."""
    import torch
    import quantized_kv_decode_gb300 as K
    w = synth.WORKLOADS["mha7b"]
    B, Hq, Hkv, D, g, S, L = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, 32, 4, w.ctx[0]
    dev = "cuda"
    rng = synth.rng_for(w.seed)
    outl = synth.outlier_channels(rng, Hkv, D)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    k, v = synth.device_kv(gen, B, L + 1, Hkv, D, outl, dev)
    q = torch.randn((B, Hq, D), generator=gen, device=dev).half()
    cap = ((L + 1 + g - 1) // g) * g
    desc = K.make_desc(4, g, Hkv, D, K.KVQ_DENSE, cap, k_per_channel=True, sink_tokens=S)
    cache = K.KVCache.allocate(desc, B, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    K.kvq_append(cache, k[:, :L].contiguous(), v[:, :L].contiguous(),
                 torch.zeros(B, dtype=torch.int32, device=dev), st)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    out = K.kvq_append_decode_attn(cache, k[:, L].contiguous(), v[:, L].contiguous(), q, lens,
                                   L + 1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    G = Hq // Hkv
    for b, kvh in ((0, 0), (B - 1, Hkv - 1), (3, 17)):
        kk = k[b, :, kvh].cpu().numpy()[None]           # [1][L+1][D]
        vv = v[b, :, kvh].cpu().numpy()[None]
        r = O.kivi_quantize(kk, vv, 4, g, S)
        S_, r0 = r["S"], r["r0"]
        assert np.array_equal(cache.k_codes[b, kvh, S_:r0].cpu().numpy(),
                              O.pack_codes(r["k_codes"][0], 4))
        assert np.array_equal(cache.k_scale[b, kvh, :r["nb"]].cpu().numpy().view(np.uint16),
                              r["k_scale"][0].view(np.uint16))
        qh = q[b, kvh * G:(kvh + 1) * G].float().cpu().numpy().astype(np.float64)
        want = O.attend(qh, r["k_hat"][0], r["v_hat"][0], 1.0 / np.sqrt(D))
        assert_close(out[b, kvh * G:(kvh + 1) * G].float().cpu().numpy(), want)


def _paged_kivi_pair(K, bits, G, g, D, lens, seed):
    """A dense and a paged axis-aware cache (4 sinks, 2 KV heads, 64-token
    pages scattered by a seeded block table) filled by the same appends."""
    import torch
    S, Hkv, page = 4, 2, 64
    Hq = Hkv * G
    B, Lmax = len(lens), max(lens)
    rng = synth.rng_for(seed)
    outl = synth.outlier_channels(rng, Hkv, D)
    k16, v16 = synth.host_kv(rng, B, Lmax + 1, Hkv, D, outl)
    q16 = synth.host_q(rng, B, Hq, D)
    need = np.maximum(np.array(lens) + 1 - S, 1)   # quantized-region tokens after the step
    mb = -(-int(max(-(-need // page))) // 4) * 4
    table, num_pages = synth.block_table(rng, need, page, max_blocks=mb, spare_pages=2)
    cap = ((Lmax + 1 + g - 1) // g) * g + g
    dd = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, cap, k_per_channel=True, sink_tokens=S)
    pd = K.make_desc(bits, g, Hkv, D, K.KVQ_PAGED, page, num_pages, table.shape[1],
                     k_per_channel=True, sink_tokens=S)
    dense = K.KVCache.allocate(dd, B)
    paged = K.KVCache.allocate(pd, B, block_table=torch.from_numpy(table))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kt, vt = torch.from_numpy(k16).cuda(), torch.from_numpy(v16).cuda()
    _fill(K, dense, kt, vt, lens, [37, 1, 64], st)
    _fill(K, paged, kt, vt, lens, [37, 1, 64], st, view_fn=_paged_view)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kn = torch.stack([kt[b, L] for b, L in enumerate(lens)]).contiguous()   # [B][Hkv][D]
    vn = torch.stack([vt[b, L] for b, L in enumerate(lens)]).contiguous()
    return dict(dense=dense, paged=paged, table=table, k16=k16, v16=v16, q16=q16, kn=kn, vn=vn,
                S=S)


@pytest.mark.parametrize("bits,G,g,D,splits", [
    (4, 1, 32, 128, 0), (8, 1, 32, 128, 0), (4, 4, 32, 128, 0), (4, 1, 16, 128, 0),
    (4, 7, 32, 64, 0), (4, 1, 32, 128, 3), (4, 4, 64, 128, 3)])
def test_kivi_paged_matches_dense(bits, G, g, D, splits):
    """Paged axis-aware caches: pages hold the tokens after the sinks, whole
    blocks per page, scattered by a seeded block table.  Filled by the same
    appends as a dense cache, the stored rows, block headers and window
    agree with the dense cache's, the fused step and a decode give the dense
    cache's outputs bit for bit (the same arithmetic: the tensor-core kernel's
    paged instances for g = 32 and 64, head_dim 64 and 128, one or several
    splits; the per-element kernel for g = 16), and both match the oracle."""
    import torch
    import quantized_kv_decode_gb300 as K
    S, Hkv, page = 4, 2, 64
    Hq = Hkv * G
    lens = [700, 35, 1300, 4]
    B, Lmax = len(lens), max(lens)
    rng = synth.rng_for(77 + bits + G + g + D + splits)
    outl = synth.outlier_channels(rng, Hkv, D)
    k16, v16 = synth.host_kv(rng, B, Lmax + 1, Hkv, D, outl)
    q16 = synth.host_q(rng, B, Hq, D)
    need = np.maximum(np.array(lens) + 1 - S, 1)   # quantized-region tokens after the step
    # rows padded to 4 entries so that one sequence's row (a view) stays
    # 16-byte aligned, as the ABI asks of every pointer
    mb = -(-int(max(-(-need // page))) // 4) * 4
    table, num_pages = synth.block_table(rng, need, page, max_blocks=mb, spare_pages=2)
    cap = ((Lmax + 1 + g - 1) // g) * g + g
    dd = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, cap, k_per_channel=True, sink_tokens=S)
    pd = K.make_desc(bits, g, Hkv, D, K.KVQ_PAGED, page, num_pages, table.shape[1],
                     k_per_channel=True, sink_tokens=S)
    dense = K.KVCache.allocate(dd, B)
    paged = K.KVCache.allocate(pd, B, block_table=torch.from_numpy(table))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kt, vt = torch.from_numpy(k16).cuda(), torch.from_numpy(v16).cuda()
    _fill(K, dense, kt, vt, lens, [37, 1, 64], st)
    _fill(K, paged, kt, vt, lens, [37, 1, 64], st, view_fn=_paged_view)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the quantized rows and K block headers, gathered through the block table
    arr = {n: (getattr(dense, n).cpu().numpy(), getattr(paged, n).cpu().numpy())
           for n in ("k_codes", "v_codes", "v_scale", "v_zero", "k_scale", "k_zero", "k_window",
                     "v_window")}
    for bi, L in enumerate(lens):
        nb = max(0, (L - S) // g)
        u = np.arange(nb * g)
        pg, off = table[bi, u // page], u % page
        for n in ("k_codes", "v_codes", "v_scale", "v_zero"):
            d, pgd = arr[n]
            assert np.array_equal(d[bi, :, S:S + nb * g], np.transpose(pgd[pg, :, off], (1, 0, 2))), n
        jb = np.arange(nb)
        for n in ("k_scale", "k_zero"):
            d, pgd = arr[n]
            got = np.transpose(pgd[table[bi, jb * g // page], :, jb % (page // g)], (1, 0, 2))
            assert np.array_equal(d[bi, :, :nb].view(np.uint16), got.view(np.uint16)), n
        for n in ("k_window", "v_window"):
            assert np.array_equal(arr[n][0][bi].view(np.uint16), arr[n][1][bi].view(np.uint16)), n
    lb = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kn = torch.stack([kt[b, L] for b, L in enumerate(lens)]).contiguous()   # [B][Hkv][D]
    vn = torch.stack([vt[b, L] for b, L in enumerate(lens)]).contiguous()
    q = torch.from_numpy(q16).cuda()
    outs = []
    for cache in (dense, paged):
        o1 = K.kvq_append_decode_attn(cache, kn, vn, q, lb, Lmax + 1, dev_status=st,
                                      num_splits=splits)
        o2 = K.kvq_decode_attn(cache, q, lb + 1, Lmax + 1, dev_status=st, num_splits=splits)
        outs.append((o1, o2))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lens1 = [L + 1 for L in lens]
    want = _oracle_out(q16, k16, v16, lens1, bits, g, S)
    (d1, d2), (p1, p2) = outs
    assert torch.equal(d1, p1) and torch.equal(d2, p2)
    for o in (d1, d2):
        assert_close(o.cpu().numpy(), want)


def test_kivi_paged_unmapped_page():
    """A block-table entry of -1 inside one sequence's quantized region: the
    decode flags KVQ_FLAG_BLOCK_TABLE and the other sequences' outputs are
    still the dense cache's, bit for bit (tensor-core paged instance, INT4
    g32, one and three splits)."""
    import torch
    import quantized_kv_decode_gb300 as K
    lens = [700, 35, 1300, 260]
    c = _paged_kivi_pair(K, 4, 1, 32, 128, lens, seed=91)
    dense, paged, table = c["dense"], c["paged"], c["table"].copy()
    table[2, 5] = -1      # rows 320-383 after the sinks of sequence 2: quantized blocks
    bad = K.KVCache(paged.desc, paged.batch, paged.k_codes, paged.v_codes, paged.k_scale,
                    paged.k_zero, paged.v_scale, paged.v_zero,
                    torch.from_numpy(table).cuda(), paged.k_window, paged.v_window)
    q = torch.from_numpy(c["q16"]).cuda()
    lb1 = torch.tensor([L + 1 for L in lens], dtype=torch.int32, device="cuda")
    for splits in (1, 3):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        want = K.kvq_decode_attn(dense, q, lb1, max(lens) + 1, dev_status=st, num_splits=splits)
        got = K.kvq_decode_attn(bad, q, lb1, max(lens) + 1, dev_status=st, num_splits=splits)
        torch.cuda.synchronize()
        assert int(st.item()) & K.KVQ_FLAG_BLOCK_TABLE
        for b in (0, 1, 3):
            assert torch.equal(got[b], want[b]), b
        assert not bool(torch.isnan(got).any())


@pytest.mark.parametrize("bits,g,S,D,Hq,Hkv,layout", [
    (4, 32, 4, 128, 32, 32, "dense"), (4, 32, 4, 128, 8, 2, "dense"), (8, 32, 0, 128, 4, 4, "dense"),
    (4, 64, 8, 128, 4, 1, "dense"), (4, 32, 3, 64, 14, 2, "dense"), (4, 32, 4, 128, 4, 4, "paged"),
    (4, 16, 1, 128, 4, 2, "dense")])
def test_kivi_one_launch_step_matches_two_calls(bits, g, S, D, Hq, Hkv, layout):
    """With one split, kvq_append_decode_attn on an axis-aware cache appends
    inside the decode launch (each (sequence, KV head) CTA writes its token's
    window slot, or quantizes the block the token completes, before it
    attends).  The cache it leaves and its output must be bit-identical to
    kvq_append followed by kvq_decode_attn, for a token landing on a sink, in
    the residual window, and completing a block (g = 16 runs the append and
    generic kernels instead)."""
    import torch
    import quantized_kv_decode_gb300 as K
    lens = [max(S - 1, 0), S + g - 1, S + 5, S + 3 * g - 1, 200]   # cached before the step
    B, Lmax = len(lens), max(lens)
    rng = synth.rng_for(501 + bits + g + S + D + Hq)
    outl = synth.outlier_channels(rng, Hkv, D)
    k16, v16 = synth.host_kv(rng, B, Lmax + 1, Hkv, D, outl)
    q16 = synth.host_q(rng, B, Hq, D)
    kt, vt = torch.from_numpy(k16).cuda(), torch.from_numpy(v16).cuda()
    kn = torch.stack([kt[b, L] for b, L in enumerate(lens)]).contiguous()   # [B][Hkv][D]
    vn = torch.stack([vt[b, L] for b, L in enumerate(lens)]).contiguous()
    q = torch.from_numpy(q16).cuda()
    lb = torch.tensor(lens, dtype=torch.int32, device="cuda")

    def fresh():
        if layout == "dense":
            cap = ((Lmax + 1 + g - 1) // g) * g + g
            desc = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, cap, k_per_channel=True, sink_tokens=S)
            cache = K.KVCache.allocate(desc, B)
            view = _seq_view
        else:
            page = 64
            need = np.maximum(np.array(lens) + 1 - S, 1)
            mb = -(-int(max(-(-need // page))) // 4) * 4
            table, num_pages = synth.block_table(synth.rng_for(9), need, page, max_blocks=mb,
                                                 spare_pages=2)
            desc = K.make_desc(bits, g, Hkv, D, K.KVQ_PAGED, page, num_pages, table.shape[1],
                               k_per_channel=True, sink_tokens=S)
            cache = K.KVCache.allocate(desc, B, block_table=torch.from_numpy(table))
            view = _paged_view
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        _fill(K, cache, kt, vt, lens, [29, 1, 64], st, view_fn=view)
        return cache, st

    two, st2 = fresh()
    K.kvq_append(two, kn[:, None].contiguous(), vn[:, None].contiguous(), lb, st2)
    o2 = K.kvq_decode_attn(two, q, lb + 1, Lmax + 1, dev_status=st2, num_splits=1)
    one, st1 = fresh()
    o1 = K.kvq_append_decode_attn(one, kn, vn, q, lb, Lmax + 1, dev_status=st1, num_splits=1)
    torch.cuda.synchronize()
    assert int(st1.item()) == 0 and int(st2.item()) == 0
    for name in ("k_codes", "v_codes", "k_scale", "k_zero", "v_scale", "v_zero", "k_window",
                 "v_window"):
        a, c = getattr(two, name), getattr(one, name)
        assert torch.equal(a.view(torch.uint8), c.view(torch.uint8)), name
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    lens1 = [L + 1 for L in lens]
    assert_close(o1.cpu().numpy(), _oracle_out(q16, k16, v16, lens1, bits, g, S))
