"""GPU parity of kvq_append: codes, scales and zeros bit-exact with the oracle."""
import numpy as np
import pytest

import oracle as O
from quantized_kv_decode_gb300 import synth
from tests._cases import Case, gpu_codes, make_inputs, oracle_step, run_gpu

pytestmark = pytest.mark.gpu


def _compare_codes(c, inp, run, ref):
    for which in ("k", "v"):
        for b in range(c.B):
            got = gpu_codes(run, c, inp, which, b)
            want = ref[(which, b)]
            if c.bits == 16:
                assert np.array_equal(got["raw"].view(np.uint16), want["raw"].view(np.uint16))
                continue
            assert np.array_equal(got["packed"], want["packed"]), (which, b)
            assert np.array_equal(got["scale"].view(np.uint16), want["scale"].view(np.uint16)), (which, b)
            assert np.array_equal(got["zero"].view(np.uint16), want["zero"].view(np.uint16)), (which, b)


@pytest.mark.parametrize("bits,g,D", [
    (4, 8, 128), (4, 16, 128), (4, 32, 128), (4, 64, 128), (4, 128, 128),
    (8, 8, 64), (8, 32, 128), (8, 64, 256), (4, 32, 64), (4, 256, 256), (16, 0, 128)])
def test_append_bit_exact_dense(bits, g, D):
    c = Case(B=3, Hq=4, Hkv=2, D=D, bits=bits, g=g, lens=np.array([37, 1, 70]), seed=bits * 100 + g)
    inp = make_inputs(c)
    run = run_gpu(c, inp)
    _, ref = oracle_step(c, inp)
    _compare_codes(c, inp, run, ref)
    assert run["status"] == 0


@pytest.mark.parametrize("bits,g,D,ps", [(4, 32, 64, 16), (8, 16, 128, 8), (4, 64, 128, 32)])
def test_append_bit_exact_paged(bits, g, D, ps):
    c = Case(B=4, Hq=4, Hkv=2, D=D, bits=bits, g=g, lens=np.array([5, 40, 17, 33]),
             layout="paged", page_size=ps, seed=7 + bits)
    inp = make_inputs(c)
    run = run_gpu(c, inp)
    _, ref = oracle_step(c, inp)
    _compare_codes(c, inp, run, ref)
    assert run["status"] == 0


def _append_direct(x16, bits, g, status_expect):
    """Append one hand-made vector per KV head and compare with the oracle."""
    import torch
    import quantized_kv_decode_gb300 as K
    B, T, Hkv, D = x16.shape
    desc = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, T)
    cache = K.KVCache.allocate(desc, B)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.from_numpy(x16).cuda()
    K.kvq_append(cache, x, x, torch.zeros(B, dtype=torch.int32, device="cuda"), st)
    torch.cuda.synchronize()
    ref = O.quantize_groups(np.transpose(x16, (0, 2, 1, 3)), bits, g)
    assert np.array_equal(cache.k_codes.cpu().numpy(), O.pack_codes(ref["codes"], bits))
    assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint16), ref["scale"].view(np.uint16))
    assert np.array_equal(cache.k_zero.cpu().numpy().view(np.uint16), ref["zero"].view(np.uint16))
    assert int(st.item()) == status_expect
    return ref


@pytest.mark.parametrize("bits", [4, 8])
def test_append_edge_groups(bits):
    """Worked group, outlier group, exact ties, constant groups, skewed groups."""
    rows = [
        [0.42, -0.13, 0.87, 0.05, -0.28, 0.61, 0.17, -0.02],
        [0.03, -0.05, 0.02, -0.01, 0.04, 0.01, -0.02, 4.80],
        list(np.array([0.0, 15.0, 2.5, 3.5, 4.5, 0.5, 1.5, 14.5]) * 2.0 ** -4),
        [0.0] * 8, [-0.0] * 8, [1.5] * 8, [-2.25] * 8, [6e-8] * 8, [65504.0] * 8, [-65504.0] * 8,
        [3.0, 3.5, 4.0, 3.25, 3.75, 3.0, 4.0, 3.5],          # all positive
        [-9.0, -8.5, -8.0, -8.75, -8.25, -9.0, -8.0, -8.5],  # all negative
        [-65504.0, 65504.0, 0.0, 1.0, -1.0, 2.0, -2.0, 3.0],
    ]
    # one KV head per row; head_dim 64 holds the 8-value group 8 times over
    x = np.tile(np.array(rows, dtype=np.float16).reshape(1, 1, len(rows), 8), (1, 1, 1, 8))
    # the all-negative group [-9, -8] has -min/s ~ 9 * 255 > 2048 at 8 bits: the
    # zero-point is clamped and flagged on both sides
    import quantized_kv_decode_gb300 as K
    flags = O.quantize_groups(np.transpose(x, (0, 2, 1, 3)), bits, 8)["flags"]
    expect = K.KVQ_FLAG_ZERO_CLAMPED if np.any(flags & O.ZERO_CLAMPED) else 0
    assert expect == (K.KVQ_FLAG_ZERO_CLAMPED if bits == 8 else 0)
    _append_direct(x, bits, 8, expect)


def test_append_flags_zero_clamped_and_nonfinite():
    x = np.zeros((1, 1, 2, 64), dtype=np.float16)
    x[0, 0, 0, :8] = [1000.0, 1000.5, 1000.0, 1000.0, 1000.0, 1000.5, 1000.0, 1000.0]
    x[0, 0, 1, 8:16] = [1.0, np.inf, 0.0, 0.5, 0.25, 0.0, 0.0, 0.0]
    x[0, 0, 1, 16:24] = np.nan
    import quantized_kv_decode_gb300 as K
    ref = _append_direct(x, 4, 8, K.KVQ_FLAG_ZERO_CLAMPED | K.KVQ_FLAG_NONFINITE)
    # flags are [B][Hkv][T][groups]
    assert ref["flags"][0, 0, 0, 0] == O.ZERO_CLAMPED
    assert ref["flags"][0, 1, 0, 1] == O.NONFINITE and ref["flags"][0, 1, 0, 2] == O.NONFINITE


def test_append_randomized_wide_ranges():
    rng = np.random.default_rng(99)
    B, T, Hkv, D = 2, 33, 3, 128
    x = rng.normal(size=(B, T, Hkv, D)) * 10.0 ** rng.uniform(-5, 3.5, size=(B, T, Hkv, 1))
    x += rng.normal(size=(B, T, Hkv, 1)) * rng.choice([0, 1, 30], size=(B, T, Hkv, 1)) * np.abs(x).max(-1, keepdims=True)
    x = np.clip(x, -6e4, 6e4).astype(np.float16)
    for bits, g in ((4, 16), (8, 32), (4, 128)):
        import torch
        import quantized_kv_decode_gb300 as K
        desc = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, T)
        cache = K.KVCache.allocate(desc, B)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        xt = torch.from_numpy(x).cuda()
        K.kvq_append(cache, xt, xt, torch.zeros(B, dtype=torch.int32, device="cuda"), st)
        torch.cuda.synchronize()
        ref = O.quantize_groups(np.transpose(x, (0, 2, 1, 3)), bits, g)
        assert np.array_equal(cache.v_codes.cpu().numpy(), O.pack_codes(ref["codes"], bits))
        assert np.array_equal(cache.v_scale.cpu().numpy().view(np.uint16), ref["scale"].view(np.uint16))
        assert np.array_equal(cache.v_zero.cpu().numpy().view(np.uint16), ref["zero"].view(np.uint16))
        flags = np.bitwise_or.reduce(ref["flags"].ravel())
        assert bool(int(st.item()) & K.KVQ_FLAG_ZERO_CLAMPED) == bool(flags & O.ZERO_CLAMPED)


def test_append_out_of_range_positions_flag_and_skip():
    import torch
    import quantized_kv_decode_gb300 as K
    rng = synth.rng_for(5)
    k, v = synth.host_kv(rng, 3, 1, 2, 64, None)
    desc = K.make_desc(4, 32, 2, 64, K.KVQ_DENSE, 8)
    cache = K.KVCache.allocate(desc, 3)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = torch.tensor([8, -1, 7], dtype=torch.int32, device="cuda")   # 8 and -1 are outside
    K.kvq_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), before, st)
    torch.cuda.synchronize()
    assert int(st.item()) == K.KVQ_FLAG_SEQ_LEN
    codes = cache.k_codes.cpu().numpy()
    assert not codes[0].any() and not codes[1].any() and codes[2, :, 7].any()
    # paged: an unmapped page flags BLOCK_TABLE and is skipped
    table = torch.tensor([[0, -1], [1, 5]], dtype=torch.int32)
    pdesc = K.make_desc(4, 32, 2, 64, K.KVQ_PAGED, 8, 2, 2)
    pc = K.KVCache.allocate(pdesc, 2, block_table=table)
    st.zero_()
    K.kvq_append(pc, torch.from_numpy(k[:2]).cuda(), torch.from_numpy(v[:2]).cuda(),
                 torch.tensor([9, 9], dtype=torch.int32, device="cuda"), st)
    torch.cuda.synchronize()
    assert int(st.item()) == K.KVQ_FLAG_BLOCK_TABLE
    assert not pc.k_codes.cpu().numpy().any()
