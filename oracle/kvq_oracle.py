"""Plain fp64 CPU oracle for low-bit KV-cache decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may use it.  It shares no code,
table or constant with the CUDA library in ``quantized_kv_decode_gb300/``;
the two meet only in the seeded synthetic inputs the tests hand to both.

Every function restates, in plain vectorised numpy, what the source pages
define.  Page titles used in the citations:

  [KVQ]   "What actually happens when you quantize a KV cache"
          (Study . Quantization, romaanj.github.io) -- sections 3-6.
  [QIO]   "Quantization & inference optimisation" (engineeratlas) --
          "Prefill, then decode", "The same output, and the work saved",
          "The KV cache, which people forget", "What the cache costs".
  [SMU]   "Serving many users at once: batching and quantization"
          (viet.sarl) -- "Batching: one read, many users".
  [CS336] "Lecture 10 . Inference" (cs336-from-scratch) -- KV-cache sizing.
  [GIB]   "Gör inference billig: KV cache, batching och kvantisering"
          (neuralialabs) -- KV-cache size per token.

Precision: all arithmetic is fp64 except the two places where a floating
point value decides an integer code (x/s and -min/s); there the oracle takes
the decision in fp32, the precision the GPU kernel uses, as required for a
bit-exact comparison.  A test pins the fp32 decision to the exact rational
decision on randomised groups.

Readings of points the pages leave open:
  * the fp16 scale is rounded UP from (max-min)/(2^b-1), the only rounding
    under which the pages' bound |x - x_hat| <= s/2 holds for every element;
  * round() is round-half-to-even, the convention of the pages' numpy/torch
    code (np.rint / torch.round);
  * the zero-point is not clamped to the code range; it is clamped to
    [-2048, 2048] (the integers fp16 holds exactly) and the group flagged
    ZERO_CLAMPED when it falls outside;
  * a constant group (max == min) uses s = |min| (1 when min == 0), so that
    every code is 0 and x_hat == min exactly;
  * a group holding inf/NaN is stored as s = z = 0, codes 0, flagged NONFINITE;
  * decode attention over an empty cache returns zeros.

Pins (tests/test_oracle_pins.py): INT2 and the NF4 levels against [KVQ]
section 7 and [GIB]'s NF4 paragraph, the axis-aware cache against the outlier
group of [KVQ] section 3 and its sink-window cost, the worked 8-value INT4
group, its
symmetric counterpart and the absmax level count of [SMU], the
outlier group of [KVQ] section 3, the byte accounting of [KVQ] section 5,
the FP16 cache sizes of [KVQ]/[QIO]/[GIB]/[CS336]/[SMU], the naive-vs-cached
work counters of [QIO], brute-force equality of cached decode and full
causal recompute, batch-vs-solo equality ([SMU]), the textbook softmax
special case, the split-K merge identity, and the round-trip error bound.
INT8 has no worked example on the pages; beyond the shared formula it is
pinned only by the error bound and exhaustive small-range brute force.
"""

from __future__ import annotations

import numpy as np

# Flag bits returned per group by quantize_groups (values are the oracle's
# own; the tests map them to the library's status word by name).
ZERO_CLAMPED = 1
NONFINITE = 2

ZERO_LIMIT = 2048  # largest |integer| such that every integer up to it is an fp16


# ---------------------------------------------------------------------------
# fp16 rounding helpers
# ---------------------------------------------------------------------------

def fp16_round_up(d: np.ndarray) -> np.ndarray:
    """Smallest fp16 value >= d, for finite d >= 0 (float64 in, float16 out).

    numpy's float64 -> float16 cast rounds to nearest-even directly from the
    double; if that landed below d the next fp16 up is taken.
    """
    d = np.asarray(d, dtype=np.float64)
    h = d.astype(np.float16)
    below = h.astype(np.float64) < d
    with np.errstate(over="ignore"):
        up = np.nextafter(h, np.float16(np.inf))
    h = np.where(below, up, h)
    return h.astype(np.float16)


# ---------------------------------------------------------------------------
# Quantizer: [KVQ] section 3 steps 2-5 and section 4
# ---------------------------------------------------------------------------

def quantize_groups(x16: np.ndarray, bits: int, group_size: int) -> dict:
    """Group-wise asymmetric uniform quantization of fp16 vectors.

    x16: float16 array [..., D]; groups are ``group_size`` consecutive
    channels of the last axis ([KVQ] section 3 step 2 groups K[3, 0:8]).

    Per group ([KVQ] section 3 step 3, section 4):
        min, max                     one pass over the group
        s = (max - min) / (2^b - 1)  the grid step, stored as fp16
        z = round(-min / s)          the code that decodes to ~0.0
        q = clamp(round(x / s) + z, 0, 2^b - 1)
    Returns dict with codes uint8 [..., D] (unpacked), scale float16 and
    zero float16 [..., D/g], flags uint32 [..., D/g].
    """
    x16 = np.asarray(x16, dtype=np.float16)
    D = x16.shape[-1]
    if D % group_size:
        raise ValueError("group_size must divide the last axis")
    ng = D // group_size
    qmax = (1 << bits) - 1
    xg16 = x16.reshape(x16.shape[:-1] + (ng, group_size))
    xg = xg16.astype(np.float64)

    finite = np.isfinite(xg).all(axis=-1)
    xg_safe = np.where(finite[..., None], xg, 0.0)

    mn = xg_safe.min(axis=-1)
    mx = xg_safe.max(axis=-1)
    r = mx - mn                       # exact: difference of two fp16 values
    d = r / qmax

    degenerate = r == 0.0
    s_regular = fp16_round_up(np.where(degenerate, 0.0, d))
    s_degenerate = np.where(mn == 0.0, 1.0, np.abs(mn)).astype(np.float16)
    s16 = np.where(degenerate, s_degenerate, s_regular).astype(np.float16)

    s32 = s16.astype(np.float32)
    # integer decisions in fp32 (x, -min and s are fp16 values, so the casts
    # are exact; the division is IEEE round-to-nearest; rint is half-even)
    z_raw = np.rint((-mn).astype(np.float32) / s32).astype(np.float64)
    clamped = np.abs(z_raw) > ZERO_LIMIT
    z = np.clip(z_raw, -ZERO_LIMIT, ZERO_LIMIT)

    t = np.rint(xg_safe.astype(np.float32) / s32[..., None]).astype(np.float64)
    q = np.clip(t + z[..., None], 0, qmax)

    flags = np.where(clamped, ZERO_CLAMPED, 0).astype(np.uint32)
    flags = np.where(finite, flags, NONFINITE).astype(np.uint32)
    s16 = np.where(finite, s16, np.float16(0.0)).astype(np.float16)
    # z is an integer code: store it without a sign on zero (rint(-0.3) is -0.0)
    z = np.where(finite, z, 0.0) + 0.0
    q = np.where(finite[..., None], q, 0.0)

    return {
        "codes": q.astype(np.uint8).reshape(x16.shape),
        "scale": s16,
        "zero": z.astype(np.float16),
        "flags": flags,
    }


def quantize_groups_symmetric(x16: np.ndarray, bits: int, group_size: int) -> dict:
    """Group-wise symmetric (absmax) uniform quantization of fp16 vectors.

    [KVQ] section 3, "Why asymmetric? A concrete comparison", sets the
    asymmetric grid against a zero-centred one whose half-width is the larger
    of |min| and |max| (s = 0.87 / 7 for the worked group).  [SMU]
    "Quantization: rounding the weights" writes that quantizer out for any
    bit width:
        qmax  = 2^(b-1) - 1
        scale = max |x| / qmax            (one scale per group, stored as fp16)
        q     = clamp(round(x / scale), -qmax - 1, qmax)
        x_hat = q * scale

    Readings: the fp16 scale is rounded up (as in the
    asymmetric quantizer) so that no element is clipped; an all-zero group
    takes s = 1 (the page's clamp_min(1e-12) scale is not an fp16 value);
    the signed q is stored as the code q + 2^(b-1), which makes the grid the
    asymmetric one with the fixed zero-point z = 2^(b-1); a group holding
    inf/NaN is stored as s = 0, code 2^(b-1) and flagged NONFINITE.

    Returns the dict of quantize_groups; "zero" holds 2^(b-1) everywhere so
    that dequantize() applies unchanged.
    """
    x16 = np.asarray(x16, dtype=np.float16)
    D = x16.shape[-1]
    if D % group_size:
        raise ValueError("group_size must divide the last axis")
    if not 2 <= bits <= 8:
        raise ValueError("bits must be in [2, 8]")
    ng = D // group_size
    qmax = (1 << (bits - 1)) - 1
    offset = 1 << (bits - 1)
    xg = x16.reshape(x16.shape[:-1] + (ng, group_size)).astype(np.float64)

    finite = np.isfinite(xg).all(axis=-1)
    xg_safe = np.where(finite[..., None], xg, 0.0)
    a = np.abs(xg_safe).max(axis=-1)                  # exact: |fp16| is an fp16 value
    s16 = np.where(a == 0.0, np.float16(1.0), fp16_round_up(a / qmax)).astype(np.float16)

    s32 = s16.astype(np.float32)
    # the integer decision in fp32, as in quantize_groups
    t = np.rint(xg_safe.astype(np.float32) / s32[..., None]).astype(np.float64)
    q = np.clip(t, -qmax - 1, qmax)
    q = np.where(finite[..., None], q, 0.0)

    flags = np.where(finite, 0, NONFINITE).astype(np.uint32)
    s16 = np.where(finite, s16, np.float16(0.0)).astype(np.float16)
    return {
        "codes": (q + offset).astype(np.uint8).reshape(x16.shape),
        "scale": s16,
        "zero": np.full(s16.shape, offset, dtype=np.float16),
        "flags": flags,
    }


def nf4_levels() -> np.ndarray:
    """The 16 normal-quantile levels of the NF4 format ([GIB], the NF4
    paragraph: levels placed at the quantiles of a normal distribution,
    dense near zero and sparse in the tails).

    Reading (the page gives no formula): level i is the (i + 1/2)/16
    quantile of N(0, 1), divided by the outermost one so that the levels
    span [-1, 1]; stored as fp16.
    """
    from scipy.special import ndtri
    z = ndtri((np.arange(16) + 0.5) / 16.0)
    return (z / z[-1]).astype(np.float16)


def quantize_groups_nf4(x16: np.ndarray, group_size: int) -> dict:
    """Block-scaled normal-quantile 4-bit quantization ([GIB], NF4).

    Per group: s = max |x| (one fp16 scale, an fp16 value already), code =
    the level nearest x / s (the quotient in fp32; ties to the lower code),
    x_hat = level[code] * s.  A group of zeros stores s = 0 (no level is 0,
    so any other s would not decode them to 0); a group holding inf/NaN
    stores s = 0 and is flagged NONFINITE.  Codes are 0 wherever s = 0.
    Returns the dict of quantize_groups with "zero" = None.
    """
    x16 = np.asarray(x16, dtype=np.float16)
    D = x16.shape[-1]
    if D % group_size:
        raise ValueError("group_size must divide the last axis")
    ng = D // group_size
    xg = x16.reshape(x16.shape[:-1] + (ng, group_size)).astype(np.float64)
    finite = np.isfinite(xg).all(axis=-1)
    xg_safe = np.where(finite[..., None], xg, 0.0)
    s16 = np.abs(xg_safe).max(axis=-1).astype(np.float16)      # exact: an fp16 value
    lv = nf4_levels().astype(np.float32)
    mids = (lv[:-1] + lv[1:]) / np.float32(2)                  # exact in fp32
    s32 = s16.astype(np.float32)
    live = s32 > 0
    with np.errstate(invalid="ignore", divide="ignore"):
        t = xg_safe.astype(np.float32) / np.where(live, s32, np.float32(1))[..., None]
    codes = np.searchsorted(mids, t, side="left")               # number of midpoints below t
    codes = np.where(live[..., None], codes, 0)
    flags = np.where(finite, 0, NONFINITE).astype(np.uint32)
    return {
        "codes": codes.astype(np.uint8).reshape(x16.shape),
        "scale": s16,
        "zero": None,
        "flags": flags,
    }


def dequantize_nf4(codes: np.ndarray, scale: np.ndarray, group_size: int) -> np.ndarray:
    """x_hat = level[code] * s in fp64 ([GIB], NF4)."""
    codes = np.asarray(codes)
    D = codes.shape[-1]
    ng = D // group_size
    lv = nf4_levels().astype(np.float64)
    qg = lv[codes.astype(np.int64)].reshape(codes.shape[:-1] + (ng, group_size))
    s = np.asarray(scale, dtype=np.float16).astype(np.float64)[..., None]
    return (qg * s).reshape(codes.shape)


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes into bytes ([KVQ] section 3 step 5, section 5).

    INT2: four codes per byte, channel 4m + k in bits 2k, 2k + 1.
    INT4: two codes per byte, even channel in the low nibble.
    INT8: one code per byte.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    if bits == 8:
        return codes.copy()
    if bits == 2:
        return (codes[..., 0::4] | (codes[..., 1::4] << 2) | (codes[..., 2::4] << 4) |
                (codes[..., 3::4] << 6)).astype(np.uint8)
    if bits != 4:
        raise ValueError("bits must be 2, 4 or 8")
    even = codes[..., 0::2]
    odd = codes[..., 1::2]
    return (even | (odd << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray, bits: int, D: int) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    if bits == 8:
        return packed.copy()
    out = np.empty(packed.shape[:-1] + (D,), dtype=np.uint8)
    if bits == 2:
        for k in range(4):
            out[..., k::4] = (packed >> (2 * k)) & 0x03
        return out
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out


def dequantize(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray,
               group_size: int) -> np.ndarray:
    """x_hat = (q - z) * s in fp64 ([KVQ] section 3 step 3, section 4)."""
    codes = np.asarray(codes)
    D = codes.shape[-1]
    ng = D // group_size
    qg = codes.astype(np.float64).reshape(codes.shape[:-1] + (ng, group_size))
    s = np.asarray(scale, dtype=np.float16).astype(np.float64)[..., None]
    z = np.asarray(zero, dtype=np.float16).astype(np.float64)[..., None]
    return ((qg - z) * s).reshape(codes.shape)


def quantize_dequantize(x16: np.ndarray, bits: int, group_size: int) -> np.ndarray:
    r = quantize_groups(x16, bits, group_size)
    return dequantize(r["codes"], r["scale"], r["zero"], group_size)


# ---------------------------------------------------------------------------
# Axis-aware (KIVI-style) cache: [KVQ] section 3 step 7 ("axis choice",
# "sinks") and section 7
# ---------------------------------------------------------------------------

def kivi_partition(L: int, sink_tokens: int, g: int) -> tuple[int, int, int]:
    """Where each of L cached positions lives.

    [KVQ] keeps the first few tokens (attention sinks) in fp16, groups K per
    channel over runs of consecutive tokens, and keeps the newest tokens that
    have not yet filled such a run in an fp16 residual window.  Returns
    (S, nb, r0): sinks are positions [0, S); quantized block j < nb covers
    [S + j g, S + (j + 1) g); the fp16 residual window is [r0, L), r0 = S + nb g,
    fewer than g tokens.
    """
    S = min(int(sink_tokens), int(L))
    nb = (int(L) - S) // g
    return S, nb, S + nb * g


def kivi_quantize(k16: np.ndarray, v16: np.ndarray, bits: int, g: int,
                  sink_tokens: int) -> dict:
    """Quantize one cache of L tokens the axis-aware way.

    k16, v16: fp16 [..., L, D].  In each quantized block of g tokens, K is
    grouped per channel: one group is one channel across the block's g
    tokens, so a hot channel shares its scale only with itself.  V is grouped
    per token, g consecutive channels of one token, as in quantize_groups.
    Both use the asymmetric quantizer of quantize_groups (only the grouping
    axis differs).  Sinks and the residual window stay fp16 (exact).

    Returns k_hat, v_hat (fp64 [..., L, D]) and the stored parts of the
    blocks: k_codes [..., nb g, D] (unpacked), k_scale / k_zero [..., nb, D],
    v_codes [..., nb g, D], v_scale / v_zero [..., nb g, D / g], flags of both.
    """
    k16 = np.asarray(k16, dtype=np.float16)
    v16 = np.asarray(v16, dtype=np.float16)
    L, D = k16.shape[-2], k16.shape[-1]
    S, nb, r0 = kivi_partition(L, sink_tokens, g)
    lead = k16.shape[:-2]
    k_hat = k16.astype(np.float64)
    v_hat = v16.astype(np.float64)
    blk_k = k16[..., S:r0, :].reshape(lead + (nb, g, D))
    # per channel: the group axis is the block's tokens
    rk = quantize_groups(np.swapaxes(blk_k, -1, -2), bits, g)           # [..., nb, D, g]
    k_codes = np.swapaxes(rk["codes"], -1, -2).reshape(lead + (nb * g, D))
    k_hat[..., S:r0, :] = np.swapaxes(
        dequantize(rk["codes"], rk["scale"], rk["zero"], g), -1, -2).reshape(lead + (nb * g, D))
    rv = quantize_groups(v16[..., S:r0, :], bits, g)
    v_hat[..., S:r0, :] = dequantize(rv["codes"], rv["scale"], rv["zero"], g)
    return {
        "k_hat": k_hat, "v_hat": v_hat, "S": S, "nb": nb, "r0": r0,
        "k_codes": k_codes, "k_scale": rk["scale"][..., 0], "k_zero": rk["zero"][..., 0],
        "k_flags": rk["flags"][..., 0],
        "v_codes": rv["codes"], "v_scale": rv["scale"], "v_zero": rv["zero"],
        "v_flags": rv["flags"],
    }


def kivi_cache_bytes(kv_heads: int, head_dim: int, tokens: int, bits: int, g: int,
                     sink_tokens: int) -> int:
    """Bytes of one layer's axis-aware cache for one sequence of ``tokens``:
    fp16 sinks and residual, and for each quantized block g code rows of K
    and V, a K header of one fp16 scale + zero per channel and a V header of
    one per group of each token."""
    S, nb, r0 = kivi_partition(tokens, sink_tokens, g)
    fp16_rows = S + (tokens - r0)
    per_block = 2 * g * head_dim * bits // 8 + 4 * head_dim + 4 * g * (head_dim // g)
    return kv_heads * (2 * 2 * head_dim * fp16_rows + nb * per_block)


# ---------------------------------------------------------------------------
# Attention: [QIO] "Prefill, then decode"; [SMU] batched decode_step
# ---------------------------------------------------------------------------

def softmax(z: np.ndarray, axis: int = -1) -> np.ndarray:
    """Max-subtracted softmax, as in the [QIO] code."""
    z = z - z.max(axis=axis, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=axis, keepdims=True)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """One decode row per query head over a cache of L rows, no mask.

    q [G][D], K and V [L][D] (fp64) -> out [G][D].
    scores = K q * scale; out = softmax(scores) V  ([QIO] decode_step).
    An empty cache (L == 0) returns zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    G, D = q.shape
    if K.shape[0] == 0:
        return np.zeros((G, D))
    scores = (q[:, None, :] * K[None, :, :]).sum(axis=-1) * scale   # [G][L]
    p = softmax(scores, axis=-1)
    return (p[:, :, None] * V[None, :, :]).sum(axis=1)              # [G][D]


def attend_partial(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Unnormalised partial over a slice of the cache: (o, m, l).

    o = sum_j exp(s_j - m) v_j, m = max_j s_j, l = sum_j exp(s_j - m).
    Empty slice -> (0, -inf, 0).  Used to pin the split-K merge.
    """
    q = np.asarray(q, dtype=np.float64)
    G, D = q.shape
    if K.shape[0] == 0:
        return np.zeros((G, D)), np.full(G, -np.inf), np.zeros(G)
    scores = (q[:, None, :] * K[None, :, :]).sum(axis=-1) * scale
    m = scores.max(axis=-1)
    e = np.exp(scores - m[:, None])
    o = (e[:, :, None] * np.asarray(V, dtype=np.float64)[None, :, :]).sum(axis=1)
    return o, m, e.sum(axis=-1)


def lse_merge(parts) -> np.ndarray:
    """Merge partials: out = sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s.

    All parts empty -> zeros.
    """
    os_ = np.stack([p[0] for p in parts])          # [S][G][D]
    ms = np.stack([p[1] for p in parts])           # [S][G]
    ls = np.stack([p[2] for p in parts])           # [S][G]
    M = ms.max(axis=0)                             # [G]
    out = np.zeros(os_.shape[1:])
    live = np.isfinite(M)
    if not live.any():
        return out
    w = np.where(np.isfinite(ms), np.exp(ms - np.where(live, M, 0.0)[None, :]), 0.0)
    num = (w[:, :, None] * os_).sum(axis=0)
    den = (w * ls).sum(axis=0)
    out[live] = num[live] / den[live, None]
    return out


def full_causal(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Masked T x T attention recomputed from scratch ([QIO] naive forward)."""
    Q = np.asarray(Q, dtype=np.float64)
    T = Q.shape[0]
    scores = Q @ np.asarray(K, dtype=np.float64).T * scale
    mask = np.triu(np.ones((T, T), dtype=bool), 1)
    scores = np.where(mask, -np.inf, scores)
    return softmax(scores, axis=-1) @ np.asarray(V, dtype=np.float64)


def decode_attention(q16: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray,
                     seq_lens, scale: float | None = None) -> np.ndarray:
    """Batched GQA decode attention over per-sequence caches ([SMU]).

    q16    [B][Hq][D]        fp16 (or float) queries
    k_hat  [B][Hkv][Lmax][D] dequantized keys (fp64)
    v_hat  [B][Hkv][Lmax][D] dequantized values
    seq_lens[b]: rows of sequence b to attend over (the new token included)
    Query head h reads KV head h // (Hq / Hkv) (contiguous grouping, as SDPA's
    enable_gqa).  scale defaults to 1/sqrt(D).  Returns fp64 [B][Hq][D].
    """
    q = np.asarray(q16).astype(np.float64)
    B, Hq, D = q.shape
    Hkv = k_hat.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        for kvh in range(Hkv):
            out[b, kvh * G:(kvh + 1) * G] = attend(
                q[b, kvh * G:(kvh + 1) * G], k_hat[b, kvh, :L], v_hat[b, kvh, :L], scale)
    return out


# ---------------------------------------------------------------------------
# Byte accounting: [QIO] "What the cache costs"; [KVQ] section 5
# ---------------------------------------------------------------------------

def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int, tokens: int,
                   bits: int, group_size: int | None = None,
                   symmetric: bool = False, nf4: bool = False) -> int:
    """Bytes of K+V cache for ``tokens`` tokens of one sequence.

    FP16 (bits == 16): 2 * layers * kv_heads * head_dim * 2 bytes per token.
    INT4/INT8: packed codes head_dim*bits/8 bytes plus a 4-byte header
    (fp16 scale + fp16 zero) per group of ``group_size`` channels; a
    symmetric group stores the 2-byte scale only ([SMU] keeps a single
    16-bit scale for each group of 32 values).
    """
    per_vector = head_dim * bits // 8
    if bits != 16:
        per_vector += (2 if (symmetric or nf4) else 4) * (head_dim // group_size)
    return 2 * layers * kv_heads * per_vector * tokens
