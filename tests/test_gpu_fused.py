"""GPU tests of kvq_append_decode_attn, the one-call decode step.

Its cache contents and status must be bit-identical to kvq_append (one
token) followed by kvq_decode_attn on the same inputs, its output must agree
with that two-call output to fp32 rounding (max |diff| <= 2e-3 is asserted
as for the oracle, and in practice it is a few fp16 ulps), and it must match
the oracle within the decode tolerance (max |err| <= 2e-3, relative L2 <=
1e-3).  Cases cover both fast kernels (INT4, INT8), head
dims 64 and 128, GQA group sizes, one and several splits, paged caches, the
new token on tile and split boundaries, and the shapes that run the append
and generic kernels in sequence (head_dim 256, fp16 cache, 16 heads per KV
head).
"""
import numpy as np
import pytest

from tests._cases import Case, assert_close, make_inputs, oracle_step, run_gpu

pytestmark = pytest.mark.gpu


def _arrays(cache):
    names = ["k_codes", "v_codes"]
    if cache.desc.bits != 16:
        names += ["k_scale", "k_zero", "v_scale", "v_zero"]
    return {n: getattr(cache, n).cpu().numpy() for n in names}


def _check_same(c, num_splits=0):
    inp = make_inputs(c)
    sep = run_gpu(c, inp, num_splits=num_splits)
    fus = run_gpu(c, inp, num_splits=num_splits, fused=True, repeat=2)
    assert fus["status"] == sep["status"] == 0
    a, b = _arrays(sep["cache"]), _arrays(fus["cache"])
    for n in a:
        assert np.array_equal(a[n].view(np.uint8), b[n].view(np.uint8)), n
    assert_close(fus["out"], sep["out"].astype(np.float64))
    # appending the same token again at the same position changes nothing
    assert np.array_equal(fus["outs"][1].view(np.uint16), fus["out"].view(np.uint16))
    ref, _ = oracle_step(c, inp)
    assert_close(fus["out"], ref)


@pytest.mark.parametrize("bits,g,D,Hq,Hkv", [
    (4, 32, 128, 4, 4), (8, 32, 128, 8, 2), (4, 64, 128, 32, 4), (4, 32, 64, 14, 2),
    (8, 8, 64, 2, 2), (4, 16, 128, 8, 8)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fused_fast_kernels(bits, g, D, Hq, Hkv, splits):
    rng = np.random.default_rng(bits * 7 + g + D + Hq)
    lens = rng.integers(1, 700, size=3)
    lens[0] = 0                                     # the new token is the only row
    c = Case(B=3, Hq=Hq, Hkv=Hkv, D=D, bits=bits, g=g, lens=lens, seed=int(lens.sum()) + 1)
    _check_same(c, splits)


@pytest.mark.parametrize("pos", [31, 32, 63, 64, 127, 128, 255, 256, 511])
def test_fused_new_token_on_tile_and_split_edges(pos):
    """pos = the new token's position; lengths make it the first or last row
    of a 32-token tile, of a warp's round of tiles, or of a split's chunk."""
    lens = np.array([pos, 511, pos + 1])
    c = Case(B=3, Hq=8, Hkv=2, D=128, bits=4, g=32, lens=lens, seed=pos)
    for s in (1, 2, 4):
        _check_same(c, s)


@pytest.mark.parametrize("ps", [16, 64])
def test_fused_paged(ps):
    lens = np.array([130, 0, 64, 47, 300])
    c = Case(B=5, Hq=14, Hkv=2, D=64, bits=4, g=32, lens=lens, seed=23, layout="paged",
             page_size=ps)
    _check_same(c, 2)
    c8 = Case(B=5, Hq=8, Hkv=2, D=128, bits=8, g=64, lens=lens, seed=24, layout="paged",
              page_size=ps)
    _check_same(c8, 0)


@pytest.mark.parametrize("bits,g,D,Hq,Hkv", [
    (4, 128, 256, 4, 1), (16, 0, 128, 8, 2), (4, 16, 128, 16, 1)])
def test_fused_two_kernel_shapes(bits, g, D, Hq, Hkv):
    lens = np.array([0, 333, 64])
    c = Case(B=3, Hq=Hq, Hkv=Hkv, D=D, bits=bits, g=g, lens=lens, seed=31 + D)
    for s in (1, 3):
        _check_same(c, s)


def test_fused_position_outside_cache_is_flagged():
    """A sequence already at capacity: SEQ_LEN is flagged, nothing is written,
    its output row is zero; the other sequence is unaffected."""
    import torch
    import quantized_kv_decode_gb300 as K
    dev = "cuda"
    cap = 64
    desc = K.make_desc(4, 32, 2, 128, K.KVQ_DENSE, cap)
    cache = K.KVCache.allocate(desc, 2, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    kv = [torch.randn((2, cap, 2, 128), generator=g, device=dev).half() for _ in range(2)]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    K.kvq_append(cache, kv[0], kv[1], torch.zeros(2, dtype=torch.int32, device=dev), st)
    before = _arrays(cache)
    kn = torch.randn((2, 2, 128), generator=g, device=dev).half()
    vn = torch.randn((2, 2, 128), generator=g, device=dev).half()
    q = torch.randn((2, 8, 128), generator=g, device=dev).half()
    lens = torch.tensor([cap, 10], dtype=torch.int32, device=dev)
    out = K.kvq_append_decode_attn(cache, kn, vn, q, lens, cap, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & K.KVQ_FLAG_SEQ_LEN
    assert not out[0].any()
    after = _arrays(cache)
    for n in before:   # sequence 0 untouched; sequence 1 changed at position 10 only
        assert np.array_equal(before[n][0], after[n][0]), n
        diff = np.nonzero((before[n][1] != after[n][1]).reshape(2, cap, -1).any(-1))[1]
        assert set(diff.tolist()) <= {10}, n
