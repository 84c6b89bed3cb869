"""GPU parity of kvq_decode_attn against the oracle on the same codes.

Tolerance (stated for fp32 accumulation): max |gpu - oracle| <= 2e-3 and
||gpu - oracle||_2 / ||oracle||_2 <= 1e-3 over all outputs of a case.
"""
import numpy as np
import pytest

from quantized_kv_decode_gb300 import synth
from tests._cases import Case, assert_close, make_inputs, oracle_step, run_gpu

pytestmark = pytest.mark.gpu


def _check(c, num_splits=0, repeat=1):
    inp = make_inputs(c)
    run = run_gpu(c, inp, num_splits=num_splits, repeat=repeat)
    ref, _ = oracle_step(c, inp)
    assert run["status"] == 0
    assert_close(run["out"], ref)
    return run, ref


def test_tiny_workload():
    """1 sequence, 4 heads = 4 KV heads, head_dim 128, context 256, INT4 group 8,
    seed 0: one decode step (the new token makes 257 rows)."""
    w = synth.WORKLOADS["tiny"]
    c = Case(B=w.batch, Hq=w.num_q_heads, Hkv=w.num_kv_heads, D=w.head_dim, bits=4,
             g=w.group_size, lens=np.array([w.ctx[0]]), seed=w.seed)
    for s in (0, 1, 2, 5):
        _check(c, num_splits=s)


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_mha_int4_g32_splits(splits):
    c = Case(B=2, Hq=4, Hkv=4, D=128, bits=4, g=32, lens=np.array([700, 451]), seed=11)
    _check(c, num_splits=splits)


@pytest.mark.parametrize("bits,g,D,Hq,Hkv", [
    (4, 64, 128, 8, 2), (4, 32, 128, 8, 2), (8, 32, 128, 8, 2), (4, 32, 64, 14, 2),
    (4, 128, 256, 4, 1), (8, 8, 64, 2, 2), (4, 16, 128, 16, 1), (16, 0, 128, 8, 2)])
def test_gqa_ragged(bits, g, D, Hq, Hkv):
    rng = np.random.default_rng(bits + g + D + Hq)
    lens = rng.integers(1, 900, size=3)
    lens[0] = 0                                  # a sequence whose only row is the new token
    c = Case(B=3, Hq=Hq, Hkv=Hkv, D=D, bits=bits, g=g, lens=lens, seed=int(lens.sum()))
    for s in (0, 1, 3):
        _check(c, num_splits=s)


@pytest.mark.parametrize("ps", [8, 16, 64])
def test_paged_matches_oracle_and_dense(ps):
    lens = np.array([130, 1, 64, 47, 300])
    dense = Case(B=5, Hq=14, Hkv=2, D=64, bits=4, g=32, lens=lens, seed=21)
    paged = Case(B=5, Hq=14, Hkv=2, D=64, bits=4, g=32, lens=lens, seed=21, layout="paged",
                 page_size=ps)
    rd, _ = _check(dense, num_splits=2)
    rp, _ = _check(paged, num_splits=2)
    assert np.array_equal(rd["out"].view(np.uint16), rp["out"].view(np.uint16))


def test_long_int8_and_int4():
    for bits in (8, 4):
        c = Case(B=1, Hq=8, Hkv=2, D=128, bits=bits, g=32, lens=np.array([5000]), seed=31)
        _check(c, num_splits=0)


def test_deterministic_run_to_run():
    c = Case(B=2, Hq=8, Hkv=2, D=128, bits=4, g=64, lens=np.array([1000, 777]), seed=41)
    run, _ = _check(c, num_splits=5, repeat=3)
    for o in run["outs"][1:]:
        assert np.array_equal(o.view(np.uint16), run["outs"][0].view(np.uint16))


def test_bad_lengths_flag_and_zero_rows():
    import torch
    import quantized_kv_decode_gb300 as K
    c = Case(B=3, Hq=4, Hkv=2, D=64, bits=4, g=32, lens=np.array([10, 20, 30]), seed=51)
    inp = make_inputs(c)
    run = run_gpu(c, inp)
    cache = run["cache"]
    q = torch.from_numpy(inp["q"]).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for splits in (1, 3):
        lens = torch.tensor([11, 10 ** 6, -4], dtype=torch.int32, device="cuda")
        out = K.kvq_decode_attn(cache, q, lens, 31, dev_status=st, num_splits=splits)
        torch.cuda.synchronize()
        assert int(st.item()) & K.KVQ_FLAG_SEQ_LEN
        o = out.cpu().numpy()
        assert not o[1].any() and not o[2].any()
        assert np.array_equal(o[0].view(np.uint16), run["out"][0].view(np.uint16))


def test_unmapped_page_flags_block_table():
    import torch
    import quantized_kv_decode_gb300 as K
    c = Case(B=2, Hq=4, Hkv=2, D=64, bits=4, g=32, lens=np.array([40, 40]), seed=61,
             layout="paged", page_size=16)
    inp = make_inputs(c)
    run = run_gpu(c, inp)
    cache = run["cache"]
    cache.block_table[1, 1] = -7                 # sequence 1 loses its second page
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = torch.tensor([41, 41], dtype=torch.int32, device="cuda")
    out = K.kvq_decode_attn(cache, torch.from_numpy(inp["q"]).cuda(), lens, 41, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == K.KVQ_FLAG_BLOCK_TABLE
    o = out.cpu().numpy()
    assert np.array_equal(o[0].view(np.uint16), run["out"][0].view(np.uint16))
    assert np.isfinite(o[1].astype(np.float32)).all()


@pytest.mark.parametrize("bits,g,D,Hq,Hkv,sym", [
    (4, 32, 128, 4, 2, False),    # 2 heads x 4 groups: 8 score columns, two group-sum levels
    (4, 64, 128, 4, 2, False),    # 2 heads x 2 groups
    (4, 64, 128, 12, 4, False),   # 3 heads padded to 4, x 2 groups
    (4, 64, 128, 16, 4, True),    # 4 heads x 2 groups, symmetric codes
    (8, 64, 128, 16, 4, False),   # INT8, 4 heads x 2 groups
    (8, 32, 128, 8, 4, True),     # INT8 symmetric, 2 heads x 4 groups
    (8, 32, 64, 8, 4, False),     # INT8 head_dim 64, 2 heads x 2 groups
    (4, 32, 64, 16, 4, False),    # head_dim 64, 4 heads x 2 groups
    (4, 32, 64, 6, 2, False),     # head_dim 64, 3 heads padded to 4
    # 16 (group, head) columns over two q n-tiles
    (4, 32, 128, 16, 4, False),   # 4 heads x 4 groups
    (4, 32, 128, 12, 4, True),    # 3 heads padded to 4, x 4 groups, symmetric codes
    (8, 32, 128, 16, 4, False),   # INT8, 4 heads x 4 groups
    (8, 16, 128, 8, 4, False),    # INT8, 2 heads x 8 groups: three group-sum levels
    (8, 16, 64, 16, 4, True),     # INT8 head_dim 64, 4 heads x 4 groups, symmetric
])
def test_token_rows_gqa(bits, g, D, Hq, Hkv, sym):
    """GQA shapes whose (group, head) pairs fit 8 or 16 score columns take
    the token-rows score layout: ragged lengths around the 32-token tile (0,
    31, 32, 33 cached tokens), several splits, and the fused step."""
    rng = np.random.default_rng(bits * 7 + g + D + Hq)
    lens = np.array([0, 31, 32, 33, int(rng.integers(300, 700))])
    c = Case(B=5, Hq=Hq, Hkv=Hkv, D=D, bits=bits, g=g, lens=lens, seed=int(lens.sum()) % 97,
             symmetric=sym)
    for s in (0, 1, 3):
        _check(c, num_splits=s)
    inp = make_inputs(c)
    run = run_gpu(c, inp, num_splits=2, fused=True)
    ref, _ = oracle_step(c, inp)
    assert run["status"] == 0
    assert_close(run["out"], ref)


def test_token_rows_gqa_paged_matches_dense():
    """The token-rows GQA layout over a paged cache gives the dense result
    bit for bit."""
    lens = np.array([130, 1, 64, 47, 300])
    dense = Case(B=5, Hq=16, Hkv=4, D=128, bits=4, g=64, lens=lens, seed=23)
    paged = Case(B=5, Hq=16, Hkv=4, D=128, bits=4, g=64, lens=lens, seed=23, layout="paged",
                 page_size=16)
    rd, _ = _check(dense, num_splits=2)
    rp, _ = _check(paged, num_splits=2)
    assert np.array_equal(rd["out"].view(np.uint16), rp["out"].view(np.uint16))


@pytest.mark.parametrize("B,Hq,Hkv,D,g,layout,fused", [
    (40, 16, 8, 128, 32, "dense", False),    # 320 CTAs: more than one wave of the SMs
    (40, 32, 8, 128, 64, "dense", True),     # fused append, token-rows GQA
    (120, 28, 4, 64, 32, "paged", False),    # 7 heads per KV head, 16-token pages
    (160, 4, 2, 64, 32, "dense", False),     # 160 sequences, one or two per length bucket
])
def test_multiwave_ragged_batches(B, Hq, Hkv, D, g, layout, fused):
    """Grids larger than one wave run the batch longest sequence first (grid
    index z is a rank in that order).  Every sequence must still get its own
    output: ragged lengths with ties, an empty context and the longest
    sequence last in the batch."""
    rng = np.random.default_rng(B + Hq + D)
    lens = rng.integers(0, 400, size=B)
    lens[:5] = 17                                # ties broken by index
    lens[5] = 0
    lens[-1] = 450                               # the longest sequence sits last
    c = Case(B=B, Hq=Hq, Hkv=Hkv, D=D, bits=4, g=g, lens=lens, seed=B % 89, layout=layout,
             page_size=16)
    inp = make_inputs(c)
    ref, _ = oracle_step(c, inp)
    for s in (0, 1):
        run = run_gpu(c, inp, num_splits=s, fused=fused)
        assert run["status"] == 0
        assert_close(run["out"], ref)


@pytest.mark.parametrize("bits,g,sym,nf4", [(4, 32, False, False), (8, 32, False, False),
                                            (2, 32, False, False), (4, 64, True, False),
                                            (4, 64, False, True)])
@pytest.mark.parametrize("k_mul,v_mul", [(8.0, 1.0), (0.05, 0.01)])
def test_magnitudes(bits, g, sym, nf4, k_mul, v_mul):
    """K and V far from N(0, 1): a sharp softmax (K x 8) and small, flat
    inputs (K x 0.05, V x 0.01).  The tensor-core kernel carries the codes
    as fp16 subnormals and the 2^24 in its scales; the outputs must still
    match the oracle on the same codes within the decode tolerance."""
    c = Case(B=2, Hq=8, Hkv=8, D=128, bits=bits, g=g, lens=np.array([1500, 333]),
             seed=5150 + bits + g, symmetric=sym, nf4=nf4)
    inp = make_inputs(c)
    for key, mul in (("k_ctx", k_mul), ("k_new", k_mul), ("v_ctx", v_mul), ("v_new", v_mul)):
        inp[key] = (inp[key].astype(np.float32) * mul).astype(np.float16)
    for fused in (False, True):
        run = run_gpu(c, inp, fused=fused)
        ref, _ = oracle_step(c, inp)
        assert run["status"] == 0
        assert_close(run["out"], ref)


@pytest.mark.parametrize("D,Hq,Hkv,layout", [
    (128, 4, 4, "dense"),    # one query head per KV head
    (128, 16, 4, "dense"),   # 4 heads per KV head
    (64, 14, 2, "dense"),    # 7 heads padded to 8, head_dim 64
    (128, 8, 2, "paged"),    # paged, 4 heads
    (64, 6, 2, "paged"),     # paged, 3 heads padded to 4, head_dim 64
])
def test_fp16_tensor_core(D, Hq, Hkv, layout):
    """fp16 caches on the tensor-core kernel (16-token tiles): lengths around
    the tile (0, 15, 16, 17 cached tokens) and a longer one, one and several
    splits, and the fused step (append kernel, then the decode)."""
    rng = np.random.default_rng(D + Hq + Hkv)
    lens = np.array([0, 15, 16, 17, int(rng.integers(300, 900))])
    c = Case(B=5, Hq=Hq, Hkv=Hkv, D=D, bits=16, g=0, lens=lens, seed=int(lens.sum()) % 89,
             layout=layout, page_size=16)
    for s in (0, 1, 3):
        _check(c, num_splits=s)
    inp = make_inputs(c)
    run = run_gpu(c, inp, num_splits=2, fused=True)
    ref, _ = oracle_step(c, inp)
    assert run["status"] == 0
    assert_close(run["out"], ref)


@pytest.mark.parametrize("g", [32, 8])  # tensor-core kernel (marked empty splits) / CUDA-core kernel
@pytest.mark.parametrize("fused", [False, True])
def test_split_workspace_needs_no_init(g, fused):
    """Split calls over a workspace filled with NaN bytes, or with bytes of a
    large finite float: sequences shorter than a split leave splits with no
    tokens, whose workspace rows the merge must not use (after the
    tensor-core kernel they carry the m = -inf marker and a stale o)."""
    lens = np.array([300, 5, 64, 0, 1000, 33, 257, 129])
    c = Case(B=8, Hq=8, Hkv=2, D=128, bits=4, g=g, lens=lens, seed=31)
    inp = make_inputs(c)
    ref, _ = oracle_step(c, inp)
    for fill in (0xFF, 0x7F):
        run = run_gpu(c, inp, num_splits=4, fused=fused, ws_fill=fill, repeat=2)
        assert run["status"] == 0
        for out in run["outs"]:
            assert np.isfinite(out).all()
            assert_close(out, ref)


@pytest.mark.parametrize("graph", [False, True])
def test_split_merge_across_calls(graph):
    """Split calls on one workspace (filled with NaN bytes first), with a new
    q before every call, eagerly or replayed from one CUDA graph: partials
    and empty-split markers left by the call before never leak into this
    call's merge (each output against the oracle for its own q)."""
    import torch
    import quantized_kv_decode_gb300 as K
    c = Case(B=3, Hq=8, Hkv=2, D=128, bits=4, g=32, lens=np.array([900, 40, 1500]), seed=41)
    inp = make_inputs(c)
    run = run_gpu(c, inp, num_splits=4)
    cache, desc = run["cache"], run["desc"]
    rows = inp["Lctx"] + 1
    assert K.kvq_decode_num_splits(desc, c.B, c.Hq, rows, 4) == 4
    lens1 = torch.from_numpy((c.lens + 1).astype(np.int32)).cuda()
    q_buf = torch.empty((c.B, c.Hq, c.D), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q_buf)
    ws = torch.full((K.kvq_decode_workspace_size(desc, c.B, c.Hq, rows, 4),), 0xFF,
                    dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        K.kvq_decode_attn(cache, q_buf, lens1, rows, out=out, workspace=ws, dev_status=status,
                          num_splits=4, stream=stream)

    rng = np.random.default_rng(5)
    step = call
    if graph:
        with torch.cuda.stream(stream):
            call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        step = g.replay
    for _ in range(3):
        q = synth.host_q(rng, c.B, c.Hq, c.D)
        q_buf.copy_(torch.from_numpy(q))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref, _ = oracle_step(c, dict(inp, q=q))
        assert_close(out.cpu().numpy(), ref)
