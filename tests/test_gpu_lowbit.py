"""GPU parity of INT2 and NF4 caches against the oracle.

INT2 packs four codes per byte (asymmetric and symmetric grids); NF4 codes
index sixteen normal-quantile levels with one absmax scale per group.  Codes
and scales must equal the oracle's bit for bit; decode attention (the CUDA-
tensor-core kernel takes INT2 at head_dim 128 with groups of 16, 32 or 64
channels, and NF4 at head_dim 64 / 128 with 2 or 4 groups per head, for up
to 8 query heads per KV head (g16 / g32 INT2: 8 / 4 (group, head) columns);
the CUDA-core kernel serves the other shapes) must match the oracle's attention over the
dequantized cache within the decode tolerance (max |err| <= 2e-3, relative
L2 <= 1e-3).  The oracle's own pins state the accuracy these formats lose.
"""
import numpy as np
import pytest

import oracle as O
from tests._cases import Case, assert_close, gpu_codes, make_inputs, oracle_step, run_gpu

pytestmark = pytest.mark.gpu


def _check(c, splits=0, fused=False):
    inp = make_inputs(c)
    run = run_gpu(c, inp, num_splits=splits, fused=fused)
    ref_out, ref = oracle_step(c, inp)
    for which in ("k", "v"):
        for b in range(c.B):
            got = gpu_codes(run, c, inp, which, b)
            want = ref[(which, b)]
            assert np.array_equal(got["packed"], want["packed"]), (which, b)
            assert np.array_equal(got["scale"].view(np.uint16), want["scale"].view(np.uint16))
            if not c.nf4 and not c.symmetric:
                assert np.array_equal(got["zero"].view(np.uint16), want["zero"].view(np.uint16))
    assert run["status"] == 0
    assert_close(run["out"], ref_out)
    return run


@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("g,D,Hq,Hkv", [(32, 128, 8, 2), (16, 64, 4, 4), (64, 128, 4, 1),
                                        (32, 128, 4, 4), (16, 128, 8, 8), (32, 128, 16, 8),
                                        (64, 128, 16, 2), (64, 128, 6, 2)])
def test_int2(sym, g, D, Hq, Hkv):
    rng = np.random.default_rng(g + D + Hq + int(sym))
    lens = rng.integers(1, 600, size=3)
    lens[0] = 0
    c = Case(B=3, Hq=Hq, Hkv=Hkv, D=D, bits=2, g=g, lens=lens, seed=int(lens.sum()), symmetric=sym)
    _check(c, 0)
    _check(c, 3, fused=True)


@pytest.mark.parametrize("g,D,Hq,Hkv", [(64, 128, 8, 2), (32, 128, 4, 4), (64, 64, 14, 2), (128, 256, 2, 1),
                                        (32, 64, 16, 2), (32, 128, 6, 2), (32, 128, 16, 2)])
def test_nf4(g, D, Hq, Hkv):
    rng = np.random.default_rng(g * 3 + D + Hq)
    lens = rng.integers(1, 700, size=3)
    lens[1] = 0
    c = Case(B=3, Hq=Hq, Hkv=Hkv, D=D, bits=4, g=g, lens=lens, seed=int(lens.sum()) + 9, nf4=True)
    _check(c, 0)
    _check(c, 2, fused=True)


@pytest.mark.parametrize("g", [16, 32, 64])
def test_int2_long_multiwave(g):
    """Tensor-core INT2: several tiles per warp, ragged tails, one and four splits."""
    lens = np.array([4095, 1, 2048, 33, 3001, 32])
    c = Case(B=6, Hq=8, Hkv=8, D=128, bits=2, g=g, lens=lens, seed=4343 + g)
    _check(c, 1, fused=True)
    _check(c, 4)


def test_int2_paged():
    lens = np.array([130, 0, 64, 47, 300])
    c = Case(B=5, Hq=8, Hkv=2, D=128, bits=2, g=64, lens=lens, seed=78, layout="paged",
             page_size=16, symmetric=True)
    _check(c, 2)
    _check(c, 0, fused=True)


def test_nf4_long_multiwave():
    """Tensor-core NF4: several tiles per warp, a ragged tail, one and four splits."""
    lens = np.array([4095, 1, 2048, 33, 3001, 32])
    c = Case(B=6, Hq=32, Hkv=8, D=128, bits=4, g=32, lens=lens, seed=4242, nf4=True)
    _check(c, 1, fused=True)
    _check(c, 4)


def test_nf4_paged():
    lens = np.array([130, 0, 64, 47, 300])
    c = Case(B=5, Hq=8, Hkv=2, D=128, bits=4, g=64, lens=lens, seed=77, layout="paged",
             page_size=16, nf4=True)
    _check(c, 2)


def test_lowbit_special_groups():
    """Zero groups, constant groups, fp16 extremes and inf/NaN (flagged)."""
    import torch
    import quantized_kv_decode_gb300 as K
    rows = [
        [0.42, -0.13, 0.87, 0.05, -0.28, 0.61, 0.17, -0.02],
        [0.0] * 8, [-0.0] * 8, [1.5] * 8, [-2.25] * 8, [6e-8] * 8, [65504.0] * 8,
        [-65504.0, 65504.0, 0.0, 1.0, -1.0, 2.0, -2.0, 3.0],
        [1.0, np.inf, 0.0, 0.5, 0.25, 0.0, 0.0, 0.0],
    ]
    x = np.tile(np.array(rows, dtype=np.float16).reshape(1, 1, len(rows), 8), (1, 1, 1, 8))
    xt = x.transpose(0, 2, 1, 3)
    for bits, kw in ((2, {}), (2, dict(symmetric=True)), (4, dict(nf4=True))):
        desc = K.make_desc(bits, 8, len(rows), 64, K.KVQ_DENSE, 1, **kw)
        cache = K.KVCache.allocate(desc, 1)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        t = torch.from_numpy(x).cuda()
        K.kvq_append(cache, t, t, torch.zeros(1, dtype=torch.int32, device="cuda"), st)
        torch.cuda.synchronize()
        if kw.get("nf4"):
            ref = O.quantize_groups_nf4(xt, 8)
        elif kw.get("symmetric"):
            ref = O.quantize_groups_symmetric(xt, bits, 8)
        else:
            ref = O.quantize_groups(xt, bits, 8)
        assert np.array_equal(cache.k_codes.cpu().numpy(), O.pack_codes(ref["codes"], bits)), kw
        assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint16), ref["scale"].view(np.uint16)), kw
        if cache.k_zero is not None:
            assert np.array_equal(cache.k_zero.cpu().numpy().view(np.uint16), ref["zero"].view(np.uint16))
        flags = int(np.bitwise_or.reduce(ref["flags"].ravel()))
        want = (K.KVQ_FLAG_NONFINITE if flags & O.NONFINITE else 0) | \
               (K.KVQ_FLAG_ZERO_CLAMPED if flags & O.ZERO_CLAMPED else 0)
        assert int(st.item()) == want, kw
