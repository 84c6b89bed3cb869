"""GPU parity of symmetric (absmax) caches against the oracle.

Symmetric caches keep one fp16 scale per group and no zero-point; the codes
are q + 2^(bits-1).  kvq_append must match quantize_groups_symmetric bit for
bit (codes and scales); kvq_decode_attn and kvq_append_decode_attn must match
the oracle's attention over the dequantized cache within the decode
tolerance (max |err| <= 2e-3, relative L2 <= 1e-3).
"""
import numpy as np
import pytest

import oracle as O
from tests._cases import Case, assert_close, gpu_codes, make_inputs, oracle_step, run_gpu

pytestmark = pytest.mark.gpu


def _check(c, num_splits=0, fused=False):
    inp = make_inputs(c)
    run = run_gpu(c, inp, num_splits=num_splits, fused=fused)
    assert run["cache"].k_zero is None and run["cache"].v_zero is None
    ref_out, ref = oracle_step(c, inp)
    for which in ("k", "v"):
        for b in range(c.B):
            got = gpu_codes(run, c, inp, which, b)
            want = ref[(which, b)]
            assert np.array_equal(got["packed"], want["packed"]), (which, b)
            assert np.array_equal(got["scale"].view(np.uint16), want["scale"].view(np.uint16))
    assert run["status"] == 0
    assert_close(run["out"], ref_out)
    return run


@pytest.mark.parametrize("bits,g,D,Hq,Hkv", [
    (4, 32, 128, 4, 4), (4, 64, 128, 8, 2), (8, 32, 128, 8, 2), (4, 32, 64, 14, 2),
    (8, 16, 64, 4, 2), (4, 8, 128, 4, 2), (8, 128, 256, 2, 1), (4, 16, 128, 16, 1)])
@pytest.mark.parametrize("splits", [0, 3])
def test_symmetric_append_and_decode(bits, g, D, Hq, Hkv, splits):
    rng = np.random.default_rng(bits * 31 + g + D + Hq)
    lens = rng.integers(1, 800, size=3)
    lens[1] = 0
    c = Case(B=3, Hq=Hq, Hkv=Hkv, D=D, bits=bits, g=g, lens=lens, seed=int(lens.sum()) + 5,
             symmetric=True)
    _check(c, splits)


@pytest.mark.parametrize("bits", [4, 8])
def test_symmetric_fused_and_paged(bits):
    lens = np.array([130, 0, 64, 47, 300])
    c = Case(B=5, Hq=8, Hkv=2, D=128, bits=bits, g=32, lens=lens, seed=61 + bits,
             layout="paged", page_size=16, symmetric=True)
    sep = _check(c, 2, fused=False)
    fus = _check(c, 2, fused=True)
    for n in ("k_codes", "v_codes", "k_scale", "v_scale"):
        assert np.array_equal(getattr(sep["cache"], n).cpu().numpy().view(np.uint8),
                              getattr(fus["cache"], n).cpu().numpy().view(np.uint8)), n


def test_symmetric_special_groups_bit_exact():
    """Zero groups, absmax ties, fp16 extremes, inf/NaN (flagged)."""
    import torch
    import quantized_kv_decode_gb300 as K
    rows = [
        [0.42, -0.13, 0.87, 0.05, -0.28, 0.61, 0.17, -0.02],
        [0.0] * 8, [-0.0] * 8, [1.5] * 8, [-2.25] * 8, [6e-8] * 8, [65504.0] * 8,
        [-65504.0, 65504.0, 0.0, 1.0, -1.0, 2.0, -2.0, 3.0],
        [7.0, -7.0, 3.5, -3.5, 0.5, -0.5, 1.5, -1.5],
        [1.0, np.inf, 0.0, 0.5, 0.25, 0.0, 0.0, 0.0],
    ]
    x = np.tile(np.array(rows, dtype=np.float16).reshape(1, 1, len(rows), 8), (1, 1, 1, 8))
    for bits in (4, 8):
        desc = K.make_desc(bits, 8, len(rows), 64, K.KVQ_DENSE, 1, symmetric=True)
        cache = K.KVCache.allocate(desc, 1)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        xt = torch.from_numpy(x).cuda()
        K.kvq_append(cache, xt, xt, torch.zeros(1, dtype=torch.int32, device="cuda"), st)
        torch.cuda.synchronize()
        ref = O.quantize_groups_symmetric(np.transpose(x, (0, 2, 1, 3)), bits, 8)
        assert np.array_equal(cache.k_codes.cpu().numpy(), O.pack_codes(ref["codes"], bits))
        assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint16), ref["scale"].view(np.uint16))
        assert int(st.item()) == K.KVQ_FLAG_NONFINITE
