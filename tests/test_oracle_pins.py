"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print (tests/golden/), exact rational arithmetic, closed forms,
invariants, and library routines for the special cases that reduce to them.
All run on CPU.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle as O


def f16(v):
    return np.asarray(v, dtype=np.float16)


# ---------------------------------------------------------------------------
# "What actually happens when you quantize a KV cache", section 3 steps 3-5
# ---------------------------------------------------------------------------

def test_worked_int4_group(golden):
    kv, rows = golden("kvq_worked_group_int4.txt")
    x = f16([float(r[1]) for r in rows])
    res = O.quantize_groups(x, kv["bits"], kv["group_size"])
    s = float(res["scale"][0])
    # min / max / range as printed (inputs are fp16-rounded, 3-decimal agreement)
    xd = x.astype(np.float64)
    assert abs(xd.min() - kv["min"]) < 5e-4
    assert abs(xd.max() - kv["max"]) < 5e-4
    # scale: range/15 = 0.07667, stored as fp16 (rounded up: within one fp16 ulp)
    assert abs(s - kv["scale"]) < 1e-4
    assert s >= (xd.max() - xd.min()) / 15
    assert abs(-xd.min() / s - kv["neg_min_over_scale"]) < 5e-3
    assert float(res["zero"][0]) == kv["zero"]
    # per-channel table: round column, code column, bits column
    for i, r in enumerate(rows):
        assert abs(float(x[i]) / s - float(r[2])) < 1e-2
        assert int(np.rint(np.float32(x[i]) / np.float32(s))) == int(r[3])
        assert int(res["codes"][i]) == int(r[4])
        assert format(int(res["codes"][i]), "04b") == r[5]
    xh = O.dequantize(res["codes"], res["scale"], res["zero"], 8)
    # the page decodes with the exact s = range/15; the stored fp16 s is at most
    # one fp16 ulp away, so x_hat may differ by |q - z| ulp plus the page's
    # 4-decimal rounding
    ulp = float(np.spacing(res["scale"][0]))
    for i, r in enumerate(rows):
        tol = abs(int(r[4]) - kv["zero"]) * ulp + 5e-5
        assert abs(xh[i] - float(r[6])) <= tol
        assert abs((xh[i] - xd[i]) - float(r[7])) <= tol + 5e-4   # x was rounded to fp16
    assert np.abs(xh - xd).max() <= kv["error_bound"]
    assert np.abs(xh - xd).max() <= s / 2


def test_worked_group_packed_bytes(golden):
    """Two codes per byte, even channel in the low nibble (step 5): the bytes
    are read off the page's bits column, odd channel's bits first."""
    kv, rows = golden("kvq_worked_group_int4.txt")
    expect = [int(rows[2 * i + 1][5] + rows[2 * i][5], 2) for i in range(4)]
    codes = np.array([int(r[4]) for r in rows], dtype=np.uint8)
    packed = O.pack_codes(codes, 4)
    assert list(packed) == expect
    assert list(O.unpack_codes(packed, 4, 8)) == list(codes)
    x = f16([float(r[1]) for r in rows])
    res = O.quantize_groups(x, 4, 8)
    assert list(O.pack_codes(res["codes"], 4)) == expect


def test_outlier_group(golden):
    kv, _ = golden("kvq_outlier_group_int4.txt")
    x = f16(kv["values"])
    res = O.quantize_groups(x, kv["bits"], kv["group_size"])
    s = float(res["scale"][0])
    assert abs(s - kv["scale"]) < 1e-3
    assert abs(15 * s - kv["range"]) < 0.01
    assert float(res["zero"][0]) == kv["zero"]
    xh = O.dequantize(res["codes"], res["scale"], res["zero"], 8)
    assert int((xh[:7] == 0.0).sum()) == kv["erased_channels"]
    assert abs(xh[7] - 4.80) <= s / 2


def test_asymmetric_step_finer_than_symmetric(golden):
    kv, _ = golden("kvq_symmetric_vs_asymmetric.txt")
    wk, rows = golden("kvq_worked_group_int4.txt")
    x = f16([float(r[1]) for r in rows])
    s = float(O.quantize_groups(x, 4, 8)["scale"][0])
    assert abs(s - kv["asymmetric_scale"]) < 1e-4
    assert abs(1 - s / kv["symmetric_scale"] - kv["finer_fraction"]) < 0.01


# ---------------------------------------------------------------------------
# Symmetric (absmax) quantizer: "What actually happens when you quantize a KV
# cache", section 3 comparison; "Serving many users at once", "Quantization:
# rounding the weights"
# ---------------------------------------------------------------------------

def test_symmetric_worked_group(golden):
    """The worked group under the symmetric grid: s = max(|min|, |max|) / 7 =
    0.124 as printed, and the asymmetric step is 38 % finer."""
    kv, _ = golden("kvq_symmetric_vs_asymmetric.txt")
    _, rows = golden("kvq_worked_group_int4.txt")
    x = f16([float(r[1]) for r in rows])
    sym = O.quantize_groups_symmetric(x, 4, 8)
    s = float(sym["scale"][0])
    assert abs(s - kv["symmetric_scale"]) < 5e-4
    a = float(np.abs(x.astype(np.float64)).max())
    assert a / 7 <= s <= float(np.nextafter(np.float16(a / 7), np.float16(np.inf))) + 1e-12
    s_asym = float(O.quantize_groups(x, 4, 8)["scale"][0])
    assert abs(1 - s_asym / s - kv["finer_fraction"]) < 0.01
    # c2 = 0.87 is the absmax: it lands on the top level 7 (code 15)
    assert int(sym["codes"][2]) == 15
    assert float(O.dequantize(sym["codes"], sym["scale"], sym["zero"], 8)[2]) == 7 * s


def test_symmetric_levels_match_page(golden):
    """2^b levels from -2^(b-1) to 2^(b-1)-1 (the page lists -2, -1, 0, 1 for
    2 bits); qmax = 127 / 7 for 8 / 4 bits; every decoded value is a level
    times the group's scale."""
    kv, rows = golden("smu_absmax_levels.txt")
    assert kv["qmax_8"] == (1 << 7) - 1 and kv["qmax_4"] == (1 << 3) - 1
    rng = np.random.default_rng(3)
    for r in rows:
        bits, levels, lo, hi = int(r[1]), int(r[2]), int(r[3]), int(r[4])
        assert levels == hi - lo + 1 == 2 ** bits
        x = f16(rng.standard_normal((64, 32)) * rng.uniform(0.01, 20, (64, 1)))
        res = O.quantize_groups_symmetric(x, bits, 32)
        q = res["codes"].astype(np.int64) - (1 << (bits - 1))
        assert q.min() >= lo and q.max() <= hi
        # the scale is rounded up, so no element is clipped: |q| <= qmax
        assert np.abs(q).max() <= hi
        xh = O.dequantize(res["codes"], res["scale"], res["zero"], 32)
        s = res["scale"].astype(np.float64)
        assert np.array_equal(xh, q.reshape(64, 1, 32).astype(np.float64).reshape(64, 32) *
                              np.repeat(s, 32, axis=-1))


def test_symmetric_scale_overhead(golden):
    """One 2-byte scale per group and no zero-point: 16 bits per 32 values on
    top of the codes, as the page states."""
    kv, _ = golden("smu_absmax_levels.txt")
    for bits in (4, 8):
        per_tok = O.kv_cache_bytes(1, 1, 128, 1, bits, kv["scale_group"], symmetric=True)
        codes = 2 * 128 * bits // 8
        assert (per_tok - codes) * 8 == 2 * (128 // kv["scale_group"]) * kv["scale_bits"]


@pytest.mark.parametrize("bits", [4, 8])
def test_symmetric_nearest_level_brute_force(bits):
    """Each code is the level nearest x / s (exhaustive over all 2^b levels,
    ties to even), decided on the fp32 quotient."""
    rng = np.random.default_rng(bits)
    x = f16(rng.standard_normal((200, 8)) * rng.uniform(0.05, 5, (200, 1)))
    res = O.quantize_groups_symmetric(x, bits, 8)
    half = 1 << (bits - 1)
    levels = np.arange(-half, half, dtype=np.float64)
    s32 = res["scale"].astype(np.float32)
    for i in range(x.shape[0]):
        t = (x[i].astype(np.float32) / s32[i, 0]).astype(np.float64)
        for k in range(8):
            d = np.abs(levels - t[k])
            best = levels[d == d.min()]
            want = best[0] if len(best) == 1 else best[np.abs(best % 2) == 0][0]
            assert int(res["codes"][i, k]) - half == int(want)


@pytest.mark.parametrize("bits", [4, 8])
def test_symmetric_is_odd_and_error_bounded(bits):
    """q(-x) = -q(x) (the grid is centred at zero; rint is symmetric), and
    |x - x_hat| <= s/2 (plus the fp32 quotient's rounding) for every element."""
    rng = np.random.default_rng(10 + bits)
    x = f16(rng.standard_normal((300, 64)) * rng.uniform(0.001, 100, (300, 1)))
    half = 1 << (bits - 1)
    a = O.quantize_groups_symmetric(x, bits, 32)
    b = O.quantize_groups_symmetric(-x, bits, 32)
    assert np.array_equal(a["scale"], b["scale"])
    assert np.array_equal(a["codes"].astype(np.int64) - half, -(b["codes"].astype(np.int64) - half))
    xh = O.dequantize(a["codes"], a["scale"], a["zero"], 32)
    s = np.repeat(a["scale"].astype(np.float64), 32, axis=-1)
    err = np.abs(xh - x.astype(np.float64))
    assert (err <= s / 2 * (1 + 1e-6) + 1e-12).all()


def test_symmetric_special_groups():
    """All-zero group: s = 1, codes at the offset, decodes to 0.  A group with
    inf/NaN: s = 0, flagged, decodes to 0.  Other groups are unaffected."""
    x = np.zeros((3, 16), dtype=np.float16)
    x[1, :] = np.float16(0.5)
    x[2, 3] = np.float16(np.inf)
    x[2, 9] = np.float16(1.0)
    res = O.quantize_groups_symmetric(x, 4, 8)
    assert float(res["scale"][0, 0]) == 1.0 and (res["codes"][0] == 8).all()
    assert res["flags"][2, 0] == O.NONFINITE and float(res["scale"][2, 0]) == 0.0
    assert res["flags"][2, 1] == 0
    xh = O.dequantize(res["codes"], res["scale"], res["zero"], 8)
    assert (xh[0] == 0).all() and (xh[2, :8] == 0).all()
    assert np.allclose(xh[1], 0.5, atol=float(res["scale"][1, 0]) / 2)
    assert abs(xh[2, 9] - 1.0) <= float(res["scale"][2, 1]) / 2 and np.isfinite(xh[2, 8:]).all()


# ---------------------------------------------------------------------------
# Lower-bit and non-uniform levels: "What actually happens when you quantize a
# KV cache", section 3 step 7 ("2-bit cliff"); "Gör inference billig", NF4
# ---------------------------------------------------------------------------

def test_int2_groups(golden):
    """Four codes and three steps per group: s = range / 3 (rounded up),
    every code in 0..3, at most four distinct decoded values, |x - x_hat|
    <= s/2; the step is range/3 against range/15 at INT4 (5x coarser)."""
    kv, _ = golden("kvq_int2.txt")
    rng = np.random.default_rng(4)
    x = f16(rng.standard_normal((200, 32)) * rng.uniform(0.01, 50, (200, 1)))
    r = O.quantize_groups(x, kv["bits"], 32)
    xd = x.astype(np.float64)
    rngs = xd.max(-1) - xd.min(-1)
    s = r["scale"][:, 0].astype(np.float64)
    assert (s * kv["steps"] >= rngs).all()
    assert (s < rngs / kv["steps"] * (1 + 2 ** -10) + 1e-12).all()
    assert r["codes"].max() == kv["codes"] - 1
    xh = O.dequantize(r["codes"], r["scale"], r["zero"], 32)
    assert max(len(set(row)) for row in xh.tolist()) <= kv["codes"]
    assert (np.abs(xh - xd) <= s[:, None] / 2 + 1e-12).all()
    s4 = O.quantize_groups(x, 4, 32)["scale"][:, 0].astype(np.float64)
    ratio = np.median(s / s4)
    assert abs(ratio - kv["int4_steps"] / kv["steps"]) < 0.05


def test_int2_pack_unpack():
    rng = np.random.default_rng(5)
    c = rng.integers(0, 4, size=(7, 64)).astype(np.uint8)
    p = O.pack_codes(c, 2)
    assert p.shape == (7, 16)
    assert int(p[0, 0]) == int(c[0, 0] | (c[0, 1] << 2) | (c[0, 2] << 4) | (c[0, 3] << 6))
    assert np.array_equal(O.unpack_codes(p, 2, 64), c)


def test_nf4_levels_shape(golden):
    """Sixteen increasing levels spanning [-1, 1], symmetric about zero,
    spaced most tightly near zero and widening toward the tails."""
    kv, _ = golden("gib_nf4.txt")
    lv = O.nf4_levels().astype(np.float64)
    assert len(lv) == kv["levels"] == 2 ** kv["code_bits"]
    assert lv[0] == -1.0 and lv[-1] == 1.0
    assert np.array_equal(lv, -lv[::-1])
    gaps = np.diff(lv)
    assert (gaps > 0).all()
    half = gaps[7:]                       # from the centre outward
    assert (np.diff(half) > 0).all()


def test_nf4_levels_are_normal_quantiles():
    """Against empirical quantiles of normal samples (numpy's generator, not
    the inverse CDF the oracle uses): level i / level 15 matches the
    (i + 1/2)/16 sample quantile over the 31/32 sample quantile."""
    x = np.random.default_rng(6).standard_normal(4_000_000)
    qs = np.quantile(x, (np.arange(16) + 0.5) / 16)
    emp = qs / qs[-1]
    lv = O.nf4_levels().astype(np.float64)
    assert np.abs(emp - lv).max() < 4e-3


def test_nf4_bits_per_value(golden):
    kv, _ = golden("gib_nf4.txt")
    D = 128
    for g, want in ((128, kv["group128_bits_per_weight"]), (64, kv["nf4_bits_per_weight"])):
        b = O.kv_cache_bytes(1, 1, D, 1, 4, g, nf4=True)
        assert b * 8 / (2 * D) == want


def test_nf4_nearest_level_and_error():
    """Each code is the level nearest x / s (brute force over all 16, ties
    to the lower code); on Gaussian blocks NF4's mean squared error is below
    that of the uniform absmax 4-bit grid at the same block size."""
    rng = np.random.default_rng(7)
    x = f16(rng.standard_normal((400, 64)))
    r = O.quantize_groups_nf4(x, 64)
    lv = O.nf4_levels().astype(np.float32)
    s32 = r["scale"].astype(np.float32)
    for i in range(0, 400, 7):
        t = x[i].astype(np.float32) / s32[i, 0]
        for k in range(64):
            d = np.abs(lv.astype(np.float64) - float(t[k]))
            assert int(r["codes"][i, k]) == int(np.argmin(d))
    xd = x.astype(np.float64)
    e_nf4 = np.mean((O.dequantize_nf4(r["codes"], r["scale"], 64) - xd) ** 2)
    sym = O.quantize_groups_symmetric(x, 4, 64)
    e_int4 = np.mean((O.dequantize(sym["codes"], sym["scale"], sym["zero"], 64) - xd) ** 2)
    assert e_nf4 < e_int4
    # the block's largest magnitude sits on a +-1 level and decodes exactly
    idx = np.abs(xd).argmax(axis=1)
    xh = O.dequantize_nf4(r["codes"], r["scale"], 64)
    assert np.array_equal(xh[np.arange(400), idx], xd[np.arange(400), idx])


def test_nf4_special_groups():
    x = np.zeros((3, 16), dtype=np.float16)
    x[1, 3] = np.float16(np.nan)
    x[2, :] = np.float16(-0.75)
    r = O.quantize_groups_nf4(x, 16)
    assert float(r["scale"][0, 0]) == 0.0 and r["flags"][0, 0] == 0
    assert float(r["scale"][1, 0]) == 0.0 and r["flags"][1, 0] == O.NONFINITE
    xh = O.dequantize_nf4(r["codes"], r["scale"], 16)
    assert (xh[:2] == 0).all()
    assert (xh[2] == -0.75).all() and (r["codes"][2] == 0).all()


# ---------------------------------------------------------------------------
# Axis-aware (KIVI-style) cache: "What actually happens when you quantize a KV
# cache", section 3 step 7 and section 7
# ---------------------------------------------------------------------------

def _outlier_tokens(golden, n_tok=8, seed=0):
    """n_tok key vectors shaped like the page's toy group: seven small
    channels and one hot channel (jittered per token)."""
    kv, _ = golden("kvq_outlier_group_int4.txt")
    base = np.array(kv["values"], dtype=np.float64)
    rng = np.random.default_rng(seed)
    k = base[None, :] * (1 + 0.5 * rng.uniform(-1, 1, (n_tok, 8)))
    return kv, f16(k)


def test_kivi_per_channel_keys_survive_outlier(golden):
    """The page's outlier group erases seven of eight channels when K is
    grouped per token; grouping per channel over the tokens keeps each
    normal channel within half its own (small) step."""
    kv, k = _outlier_tokens(golden)
    per_token = O.quantize_groups(k, 4, 8)
    xh = O.dequantize(per_token["codes"], per_token["scale"], per_token["zero"], 8)
    assert ((xh[:, :7] == 0.0).sum(axis=1) == kv["erased_channels"]).all()
    r = O.kivi_quantize(k, k, 4, 8, sink_tokens=0)
    assert r["nb"] == 1 and r["S"] == 0 and r["r0"] == 8
    kd = k.astype(np.float64)
    err = np.abs(r["k_hat"] - kd)
    s_ch = r["k_scale"][0].astype(np.float64)                      # one scale per channel
    assert (err <= s_ch[None, :] / 2 + 1e-12).all()
    assert (s_ch[:7] < 0.02).all() and s_ch[7] > 0.05              # only the hot channel is coarse
    assert (r["k_hat"][:, :7] != 0.0).sum() >= 50                  # normal channels not erased
    assert err[:, :7].max() < 0.2 * np.abs(kd[:, :7]).max()


def test_kivi_partition_and_fp16_parts():
    """Sinks and the residual window are stored exactly; blocks cover whole
    runs of g tokens after the sinks."""
    rng = np.random.default_rng(1)
    g, S = 16, 3
    for L in (0, 2, 3, 3 + 15, 3 + 16, 3 + 16 * 3 + 5, 200):
        k = f16(rng.standard_normal((2, L, 32)))
        v = f16(rng.standard_normal((2, L, 32)))
        r = O.kivi_quantize(k, v, 4, g, S)
        S_, nb, r0 = O.kivi_partition(L, S, g)
        assert (r["S"], r["nb"], r["r0"]) == (S_, nb, r0)
        assert S_ == min(S, L) and r0 == S_ + nb * g and 0 <= L - r0 < g
        for part in (slice(0, S_), slice(r0, L)):
            assert np.array_equal(r["k_hat"][:, part], k[:, part].astype(np.float64))
            assert np.array_equal(r["v_hat"][:, part], v[:, part].astype(np.float64))
        if nb:
            assert not np.array_equal(r["k_hat"][:, S_:r0], k[:, S_:r0].astype(np.float64))


def test_kivi_grouping_axes():
    """Axis checks that a transposed grouping would fail: permuting tokens
    inside a block permutes K codes and leaves the per-channel K scales
    alone, while V scales follow their tokens; permuting channels permutes
    the K scales."""
    rng = np.random.default_rng(2)
    g, D = 8, 16
    k = f16(rng.standard_normal((g, D)) * rng.uniform(0.1, 10, (1, D)))
    v = f16(rng.standard_normal((g, D)) * rng.uniform(0.1, 10, (g, 1)))
    r = O.kivi_quantize(k, v, 4, g, 0)
    perm = rng.permutation(g)
    rp = O.kivi_quantize(k[perm], v[perm], 4, g, 0)
    assert np.array_equal(rp["k_scale"], r["k_scale"]) and np.array_equal(rp["k_zero"], r["k_zero"])
    assert np.array_equal(rp["k_codes"], r["k_codes"][perm])
    assert np.array_equal(rp["v_scale"], r["v_scale"][perm])
    cperm = rng.permutation(D)
    rc = O.kivi_quantize(k[:, cperm], v, 4, g, 0)
    assert np.array_equal(rc["k_scale"][0], r["k_scale"][0][cperm])
    # K scale per channel from that channel's range over the block's tokens
    rngs = k.astype(np.float64).max(0) - k.astype(np.float64).min(0)
    assert (r["k_scale"][0].astype(np.float64) * 15 >= rngs).all()


@pytest.mark.parametrize("bits", [4, 8])
def test_kivi_error_bound(bits):
    rng = np.random.default_rng(20 + bits)
    g, S, L, D = 32, 4, 4 + 32 * 5 + 7, 64
    k = f16(rng.standard_normal((3, L, D)) * np.where(np.arange(D) % 17 == 0, 10.0, 1.0))
    v = f16(rng.standard_normal((3, L, D)))
    r = O.kivi_quantize(k, v, bits, g, S)
    ks = np.repeat(r["k_scale"].astype(np.float64), g, axis=-2)           # [3][nb g][D]
    assert (np.abs(r["k_hat"][:, S:r["r0"]] - k[:, S:r["r0"]]) <= ks / 2 + 1e-12).all()
    vs = np.repeat(r["v_scale"].astype(np.float64), g, axis=-1)
    assert (np.abs(r["v_hat"][:, S:r["r0"]] - v[:, S:r["r0"]]) <= vs / 2 + 1e-12).all()


def test_kivi_fp16_window_cost(golden):
    """A 128-token fp16 window next to a 4096-token cache costs about 3 % of
    the fp16 cache; the window bytes do not grow with the context."""
    kv, _ = golden("kvq_sink_window.txt")
    acc, _ = golden("kvq_byte_accounting.txt")
    H, D = acc["kv_heads"], acc["head_dim"]
    w = kv["window_tokens"]
    window = O.kivi_cache_bytes(H, D, w, 4, 128, sink_tokens=w)        # all fp16
    full = O.kv_cache_bytes(1, H, D, kv["ctx_tokens"], 16)
    assert window == O.kv_cache_bytes(1, H, D, w, 16)
    assert abs(window / full - kv["window_cost_fraction"]) < 0.005
    # quantized blocks cost what per-token INT4 costs, with one header per channel
    q = O.kivi_cache_bytes(H, D, 128, 4, 128, sink_tokens=0)
    assert q == O.kv_cache_bytes(1, H, D, 128, 4, 128)


# ---------------------------------------------------------------------------
# Closed forms and exact arithmetic
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [4, 8])
def test_exact_grid_roundtrip(bits):
    """Values on an exactly representable grid spanning 2^b - 1 steps are
    reproduced exactly, with the codes equal to the grid indices."""
    qmax = (1 << bits) - 1
    step = 2.0 ** -6
    rng = np.random.default_rng(7)
    for offset in (-100, -3, 0, 17, qmax // 2):
        idx = np.concatenate([[0, qmax], rng.integers(0, qmax + 1, size=6)])
        x = f16((idx - offset) * step)
        res = O.quantize_groups(x, bits, 8)
        assert float(res["scale"][0]) == step
        assert float(res["zero"][0]) == offset
        assert list(res["codes"]) == list(idx)
        assert np.array_equal(O.dequantize(res["codes"], res["scale"], res["zero"], 8),
                              x.astype(np.float64))


def _exact_codes(x16, bits, s16):
    """Rational-arithmetic codes for one group (Python round() is half-even)."""
    qmax = (1 << bits) - 1
    xs = [Fraction(float(v)) for v in x16]
    s = Fraction(float(s16))
    z = round(-min(xs) / s)
    z = max(-O.ZERO_LIMIT, min(O.ZERO_LIMIT, z))
    return [max(0, min(qmax, round(v / s) + z)) for v in xs], z


@pytest.mark.parametrize("bits", [4, 8])
def test_fp32_decisions_equal_exact_rounding(bits):
    """The fp32 x/s and -min/s decisions give the codes exact arithmetic gives."""
    rng = np.random.default_rng(11 + bits)
    groups = []
    for _ in range(600):
        scale = 10.0 ** rng.uniform(-3, 2)
        center = rng.normal() * scale * rng.choice([0.0, 1.0, 20.0])
        groups.append(rng.normal(size=8) * scale + center)
    # exact ties x/s = k + 1/2 with s = 2^-4
    base = np.array([0.0, 15.0, 2.5, 3.5, 4.5, 0.5, 1.5, 14.5]) * 2.0 ** -4
    groups.append(base if bits == 4 else np.concatenate([[0.0, 255.0], base[2:] * 16]) * 2.0 ** -4)
    x16 = f16(np.stack(groups))
    res = O.quantize_groups(x16, bits, 8)
    for i in range(x16.shape[0]):
        codes, z = _exact_codes(x16[i], bits, res["scale"][i, 0])
        assert list(res["codes"][i]) == codes, i
        assert float(res["zero"][i, 0]) == z


def test_ties_round_half_even():
    x = f16(np.array([0.0, 15.0, 2.5, 3.5, 4.5, 0.5, 1.5, 14.5]) * 2.0 ** -4)
    res = O.quantize_groups(x, 4, 8)
    assert float(res["scale"][0]) == 2.0 ** -4
    assert list(res["codes"]) == [0, 15, 2, 4, 4, 0, 2, 14]


def test_fp16_round_up_is_smallest_upper_bound():
    rng = np.random.default_rng(3)
    d = np.concatenate([10.0 ** rng.uniform(-9, 4.5, size=20000),
                        np.array([0.0, 2.0 ** -24, 1.0, 65504.0, 2.0 ** -14])])
    h = O.fp16_round_up(d)
    hd = h.astype(np.float64)
    assert np.all(hd >= d)
    below = np.nextafter(h, np.float16(-np.inf)).astype(np.float64)
    assert np.all((below < d) | (hd == 0.0))
    exact = f16(rng.normal(size=1000)).astype(np.float64)
    assert np.array_equal(O.fp16_round_up(np.abs(exact)).astype(np.float64), np.abs(exact))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("g", [8, 16, 32, 64, 128])
def test_roundtrip_error_bound(bits, g):
    """|x - x_hat| <= s/2 for every element of every unflagged group
    ("What actually happens when you quantize a KV cache", section 4)."""
    rng = np.random.default_rng(bits * 1000 + g)
    D = 128 if g <= 128 else g
    rows = [rng.normal(size=(64, D)),
            rng.normal(size=(16, D)) * 10.0 ** rng.uniform(-4, 2, size=(16, 1)),
            np.abs(rng.normal(size=(16, D))) + 3.0,         # all-positive groups
            -np.abs(rng.normal(size=(16, D))) - 0.5,        # all-negative groups
            rng.standard_cauchy(size=(16, D)).clip(-6e4, 6e4)]
    x16 = f16(np.concatenate(rows))
    res = O.quantize_groups(x16, bits, g)
    ok = res["flags"] == 0
    xh = O.dequantize(res["codes"], res["scale"], res["zero"], g)
    err = np.abs(xh - x16.astype(np.float64)).reshape(x16.shape[0], D // g, g).max(-1)
    half = res["scale"].astype(np.float64) / 2
    assert ok.mean() > 0.9
    assert np.all(err[ok] <= half[ok])


def test_degenerate_constant_groups():
    vals = [0.0, -0.0, 1.5, -2.25, 6e-8, -6e-8, 65504.0, -65504.0]
    x16 = f16(np.repeat(np.array(vals)[:, None], 8, axis=1))
    res = O.quantize_groups(x16, 4, 8)
    assert np.all(res["codes"] == 0)
    assert np.all(res["flags"] == 0)
    xh = O.dequantize(res["codes"], res["scale"], res["zero"], 8)
    assert np.array_equal(xh, x16.astype(np.float64))


def test_zero_point_outside_fp16_integers_is_clamped_and_flagged():
    x16 = f16([[1000.0, 1000.5, 1000.0, 1000.0, 1000.0, 1000.5, 1000.0, 1000.0]])
    res = O.quantize_groups(x16, 4, 8)
    assert res["flags"][0, 0] == O.ZERO_CLAMPED
    assert float(res["zero"][0, 0]) == -O.ZERO_LIMIT


def test_zero_point_is_an_integer_without_signed_zero():
    """z is the integer code that decodes to ~0.0 ("What actually happens when
    you quantize a KV cache", section 3 step 3): -min/s in (-1/2, 0) rounds to
    the integer 0, stored as +0."""
    x16 = f16([[0.01, 0.5, 0.6, 0.7, 0.8, 0.9, 1.0, 1.1],
               [-0.01, -0.5, -0.6, -0.7, -0.8, -0.9, -1.0, -0.02]])
    res = O.quantize_groups(x16, 4, 8)
    assert int(res["zero"][0, 0].view(np.uint16)) == 0
    assert not np.any(res["zero"].view(np.uint16) == 0x8000)
    rng = np.random.default_rng(1)
    many = f16(np.abs(rng.normal(size=(2000, 8))) + rng.uniform(0, 3, size=(2000, 1)))
    assert not np.any(O.quantize_groups(many, 4, 8)["zero"].view(np.uint16) == 0x8000)


def test_nonfinite_group_is_zeroed_and_flagged():
    x16 = f16([[1.0, np.inf, 0.0, 0.5, 0.25, 0.0, 0.0, 0.0],
               [1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0]])
    res = O.quantize_groups(x16, 4, 8)
    assert res["flags"][0, 0] == O.NONFINITE and res["flags"][1, 0] == 0
    assert float(res["scale"][0, 0]) == 0.0 and float(res["zero"][0, 0]) == 0.0
    assert np.all(res["codes"][0] == 0)


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_unpack_identity(bits):
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 1 << bits, size=(7, 64), dtype=np.uint8)
    packed = O.pack_codes(codes, bits)
    assert packed.shape[-1] == 64 * bits // 8
    assert np.array_equal(O.unpack_codes(packed, bits, 64), codes)


# ---------------------------------------------------------------------------
# Byte accounting
# ---------------------------------------------------------------------------

def test_fp16_cache_sizes(golden):
    _, rows = golden("fp16_cache_sizes.txt")
    assert len(rows) >= 10
    for r in rows:
        layers, kvh, hd, nbytes, tokens, expect, tol = map(int, r[2:9])
        assert nbytes == 2
        got = O.kv_cache_bytes(layers, kvh, hd, tokens, 16)
        assert abs(got - expect) <= tol, r[1]


def test_quantized_byte_accounting(golden):
    kv, rows = golden("kvq_byte_accounting.txt")
    L, H, D = kv["layers"], kv["kv_heads"], kv["head_dim"]
    assert O.kv_cache_bytes(1, H, D, 1, 16) == kv["fp16_bytes_per_token_per_layer"]
    # one 128-channel group record: 64 B of codes + 4 B header
    assert O.kv_cache_bytes(1, 1, 128, 1, 4, 128) // 2 == kv["group128_record_bytes"]
    assert O.kv_cache_bytes(1, 1, 128, 1, 16) // 2 == kv["group128_fp16_bytes"]
    fp16 = O.kv_cache_bytes(L, H, D, 1, 16)
    int4 = O.kv_cache_bytes(L, H, D, 1, 4, 128)
    assert fp16 == kv["fp16_element_bytes_per_token"] == kv["fp16_total_per_token_kib"] * 1024
    groups = 2 * L * H * (D // 128)
    assert groups == kv["int4_g128_header_groups_per_token"]
    assert groups * 4 == kv["int4_g128_header_bytes_per_token"]
    assert int4 - groups * 4 == kv["int4_g128_element_bytes_per_token"]
    assert int4 == kv["int4_g128_total_per_token_kib"] * 1024
    T = kv["seq_tokens"]
    assert O.kv_cache_bytes(L, H, D, T, 16) == kv["fp16_seq_gib"] * 2 ** 30
    assert O.kv_cache_bytes(L, H, D, T, 4, 128) == kv["int4_g128_seq_mib"] * 2 ** 20
    for r in rows:
        g, hdr_bits, eff_bits, ratio = int(r[1]), float(r[2]), float(r[3]), float(r[4])
        per_tok = O.kv_cache_bytes(L, H, D, 1, 4, g)
        values = 2 * L * H * D
        assert abs(per_tok * 8 / values - eff_bits) < 1e-9
        assert abs(per_tok * 8 / values - 4 - hdr_bits) < 1e-9
        assert abs(fp16 / per_tok - ratio) < 0.005


# ---------------------------------------------------------------------------
# Attention: cached decode vs recompute, batching, GQA, split merge
# ---------------------------------------------------------------------------

def _toy_model(d, vocab, seed):
    rng = np.random.default_rng(seed)
    E = rng.normal(size=(vocab, d))
    Wq, Wk, Wv, Wo = (rng.normal(size=(d, d)) * 0.1 for _ in range(4))
    Wlm = rng.normal(size=(d, vocab)) * 0.1
    return E, Wq, Wk, Wv, Wo, Wlm


def test_append_then_attend_work_counters(golden):
    """Naive re-forward vs prefill+decode through the oracle's attention:
    same tokens, and the page's work counters -- which hold only if each
    decode step scores every cached row including the one just appended."""
    kv, _ = golden("decode_work_counters.txt")
    d, vocab = 16, 64
    E, Wq, Wk, Wv, Wo, Wlm = _toy_model(d, vocab, 0)
    scale = 1.0 / np.sqrt(d)
    prompt = [5, 9, 2, 41][:kv["prompt_tokens"]]
    n_new = kv["new_tokens"]

    work = {"proj": 0, "scores": 0}

    def forward(tokens):
        x = E[tokens]
        work["proj"] += 3 * len(tokens)
        work["scores"] += len(tokens) ** 2
        ctx = O.full_causal(x @ Wq, x @ Wk, x @ Wv, scale)
        return (ctx @ Wo) @ Wlm

    tokens = list(prompt)
    for _ in range(n_new):
        tokens.append(int(np.argmax(forward(tokens)[-1])))
    naive_tokens, naive = tokens, dict(work)

    work = {"proj": 0, "scores": 0}
    x = E[prompt]
    cache_k, cache_v = x @ Wk, x @ Wv
    work["proj"] += 3 * len(prompt)
    work["scores"] += len(prompt) ** 2
    logits = ((O.full_causal(x @ Wq, cache_k, cache_v, scale) @ Wo) @ Wlm)[-1]
    tokens = list(prompt)
    for _ in range(n_new):
        nxt = int(np.argmax(logits))
        tokens.append(nxt)
        e = E[nxt]
        q, k, v = e @ Wq, e @ Wk, e @ Wv
        work["proj"] += 3
        cache_k = np.vstack([cache_k, k])
        cache_v = np.vstack([cache_v, v])
        work["scores"] += cache_k.shape[0]
        ctx = O.attend(q[None], cache_k, cache_v, scale)[0]
        logits = (ctx @ Wo) @ Wlm
    cached = dict(work)

    assert tokens == naive_tokens
    assert naive == {"proj": kv["naive_proj"], "scores": kv["naive_scores"]}
    assert cached == {"proj": kv["cached_proj"], "scores": kv["cached_scores"]}


@pytest.mark.parametrize("T,D", [(1, 4), (5, 8), (16, 8), (9, 3)])
def test_decode_row_equals_full_causal_last_row(T, D):
    rng = np.random.default_rng(T * 31 + D)
    Q, K, V = (rng.normal(size=(T, D)) for _ in range(3))
    scale = 1.0 / np.sqrt(D)
    full = O.full_causal(Q, K, V, scale)
    for t in range(1, T + 1):
        row = O.attend(Q[t - 1:t], K[:t], V[:t], scale)[0]
        assert np.abs(row - full[t - 1]).max() <= 1e-12


def test_batch_equals_solo_runs():
    rng = np.random.default_rng(2)
    B, Hq, Hkv, D, Lmax = 3, 4, 2, 8, 12
    q = rng.normal(size=(B, Hq, D))
    K = rng.normal(size=(B, Hkv, Lmax, D))
    V = rng.normal(size=(B, Hkv, Lmax, D))
    lens = [12, 1, 7]
    batched = O.decode_attention(q, K, V, lens)
    for b in range(B):
        solo = O.decode_attention(q[b:b + 1], K[b:b + 1], V[b:b + 1], [lens[b]])
        assert np.array_equal(batched[b], solo[0])


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 1), (8, 2), (14, 2)])
def test_gqa_matches_sdpa_enable_gqa(Hq, Hkv):
    """Special case reducing to a library routine: PyTorch's fp64 CPU
    scaled_dot_product_attention with enable_gqa, the call the batched
    decode step of "Serving many users at once" makes."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(Hq * 10 + Hkv)
    B, D, L = 2, 16, 9
    q = rng.normal(size=(B, Hq, D))
    K = rng.normal(size=(B, Hkv, L, D))
    V = rng.normal(size=(B, Hkv, L, D))
    ours = O.decode_attention(q, K, V, [L] * B)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None, :], torch.from_numpy(K), torch.from_numpy(V),
        enable_gqa=True)[:, :, 0, :].numpy()
    assert np.abs(ours - ref).max() <= 1e-12


def test_textbook_softmax_special_case():
    """G = 1: softmax(q K^T / sqrt(d)) V with scipy's softmax."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(9)
    q, K, V = rng.normal(size=(1, 32)), rng.normal(size=(40, 32)), rng.normal(size=(40, 32))
    ref = special.softmax(K @ q[0] / np.sqrt(32)) @ V
    assert np.abs(O.attend(q, K, V, 1 / np.sqrt(32))[0] - ref).max() <= 1e-12


@pytest.mark.parametrize("S", [1, 2, 3, 7])
def test_split_merge_equals_single_pass(S):
    rng = np.random.default_rng(S)
    G, D, L = 3, 16, 50
    q, K, V = rng.normal(size=(G, D)), rng.normal(size=(L, D)) * 3, rng.normal(size=(L, D))
    scale = 1 / 4
    cuts = np.sort(rng.integers(0, L + 1, size=S - 1))
    bounds = [0, *cuts.tolist(), L]          # partitions may contain empty slices
    parts = [O.attend_partial(q, K[a:b], V[a:b], scale) for a, b in zip(bounds[:-1], bounds[1:])]
    assert np.abs(O.lse_merge(parts) - O.attend(q, K, V, scale)).max() <= 1e-12


def test_empty_cache_gives_zeros():
    q = np.ones((2, 4))
    assert np.array_equal(O.attend(q, np.zeros((0, 4)), np.zeros((0, 4)), 0.5), np.zeros((2, 4)))
    parts = [O.attend_partial(q, np.zeros((0, 4)), np.zeros((0, 4)), 0.5)] * 3
    assert np.array_equal(O.lse_merge(parts), np.zeros((2, 4)))
