"""Seeded random sweep of decode shapes against the oracle.

Each case draws a combination the hand-written cases may not meet:
- a cache format: INT2, INT4, INT8 (asymmetric or symmetric), NF4 or fp16;
- head_dim 64 or 128, and a group size the format allows;
- 1-16 query heads per KV head;
- a dense or paged layout;
- ragged lengths around the 32-token tile (0, 1, 31, 32, 33, random);
- a split count and the fused or two-call step.

The tensor-core, CUDA-core and merge paths all appear.  The bar is the decode
tolerance: max |err| <= 2e-3 and relative L2 <= 1e-3.  Shapes the library
reports as unsupported are skipped.
"""
import numpy as np
import pytest

from tests._cases import Case, assert_close, make_inputs, oracle_step, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 40


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    fmt = rng.choice(["int4", "int4", "int4", "int8", "int8", "int2", "nf4", "fp16"])
    sym = bool(fmt in ("int2", "int4", "int8") and rng.random() < 0.3)
    D = int(rng.choice([64, 128]))
    if fmt == "fp16":
        bits, g = 16, 0
    elif fmt == "nf4":
        bits, g = 4, int(rng.choice([32, 64]))
    elif fmt == "int2":
        bits, g = 2, int(rng.choice([16, 32, 64]))
    else:
        bits = 4 if fmt == "int4" else 8
        g = int(rng.choice([8, 16, 32, 64] if bits == 4 else [16, 32, 64]))
    G = int(rng.choice([1, 1, 2, 3, 4, 7, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 5))
    lens = np.array([int(rng.choice([0, 1, 31, 32, 33, int(rng.integers(2, 600))]))
                     for _ in range(B)])
    layout = "paged" if (bits in (4, 8) and fmt != "nf4" and rng.random() < 0.35) else "dense"
    page = int(rng.choice([8, 16, 32]))
    splits = int(rng.choice([0, 0, 1, 3]))
    fused = bool(rng.random() < 0.5)
    c = Case(B=B, Hq=G * Hkv, Hkv=Hkv, D=D, bits=bits, g=g, lens=lens, layout=layout,
             page_size=page, seed=2000 + i, symmetric=sym, nf4=(fmt == "nf4"))
    return c, splits, fused


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_oracle(i):
    import quantized_kv_decode_gb300 as K
    c, splits, fused = _draw(i)
    inp = make_inputs(c)
    try:
        run = run_gpu(c, inp, num_splits=splits, fused=fused)
    except K.KVQError as e:
        if "UNSUPPORTED" in str(e):
            pytest.skip(f"unsupported shape: {e}")
        raise
    ref, _ = oracle_step(c, inp)
    assert run["status"] == 0
    assert_close(run["out"], ref)
