// Group-wise asymmetric quantization of fp16 vectors, shared by the append
// kernel and the fused append + decode path.
//
// "What actually happens when you quantize a KV cache", section 3 steps 2-5
// and section 4: per group of g channels, min and max, an fp16 scale and an
// integer zero-point, codes clamp(round(x/s) + z, 0, 2^b - 1), two INT4
// codes per byte with the even channel in the low nibble.
//
// Arithmetic (fixed so that codes are reproducible bit for bit):
//   range = max - min            fp64 (exact for two fp16 values)
//   s     = the smallest fp16 with s * (2^b - 1) >= range (range / (2^b - 1)
//           rounded toward +inf): an fp32 estimate, then exact fp64 checks
//   z     = rint(-min / s)       fp32 IEEE division, round half to even,
//                                clamped to +-2048 (flagged) and stored as an
//                                integer (+0, never -0)
//   q     = clamp(rint(x / s) + z, 0, 2^b - 1)
//   constant group: s = |min| (1 when min = 0), so every code is 0 and the
//   value decodes exactly; a group holding inf/NaN: s = z = 0, codes 0, flagged.
// Translation units including this file must not use fast-math: '/' stays div.rn.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

namespace quant_detail {

__device__ __forceinline__ double half_bits_value(unsigned short h) {
  return (double)__half2float(__ushort_as_half(h));
}

// smallest fp16 s > 0 with s * qmax >= range, for 0 < range <= 2 * 65504
__device__ __forceinline__ __half scale_round_up(double range, int qmax) {
  unsigned short h;
  const float est = (float)range / (float)qmax;
  asm("cvt.rp.f16.f32 %0, %1;" : "=h"(h) : "f"(est));
  // the estimate is within one fp16 step of the answer; settle it exactly
  // (h * qmax is exact in fp64: 11-bit significand times an 8-bit integer)
  if (half_bits_value(h) * qmax < range) h = (unsigned short)(h + 1);
  if (h > 1 && half_bits_value((unsigned short)(h - 1)) * qmax >= range)
    h = (unsigned short)(h - 1);
  return __ushort_as_half(h);
}

}  // namespace quant_detail

// Parameters of one asymmetric group from its min and max (fp16 values as
// fp32) and whether all its values were finite.
struct GroupParams {
  __half s, z;     // stored scale and zero-point
  float sf, zf;    // the same as fp32 (zf an integer)
  uint32_t flags;  // KVQ_FLAG_ZERO_CLAMPED / KVQ_FLAG_NONFINITE
  bool finite;
};

template <int BITS>
__device__ __forceinline__ GroupParams group_params(float mn, float mx, bool finite) {
  constexpr int QMAX = (1 << BITS) - 1;
  GroupParams r;
  r.s = __ushort_as_half(0);
  r.z = __ushort_as_half(0);
  r.sf = 0.f;
  r.zf = 0.f;
  r.flags = 0;
  r.finite = finite;
  if (!finite) {
    r.flags = KVQ_FLAG_NONFINITE;
    return r;
  }
  const double range = (double)mx - (double)mn;
  if (range == 0.0) {
    r.s = __float2half_rn(mn == 0.f ? 1.f : fabsf(mn));
  } else {
    r.s = quant_detail::scale_round_up(range, QMAX);
  }
  r.sf = __half2float(r.s);
  float zf = rintf(__fdiv_rn(-mn, r.sf));
  if (fabsf(zf) > 2048.f) {
    r.flags |= KVQ_FLAG_ZERO_CLAMPED;
    zf = fminf(fmaxf(zf, -2048.f), 2048.f);
  }
  r.zf = zf;
  r.z = __int2half_rn((int)zf);
  return r;
}

// The code of one value x of a group: clamp(rint(x / s) + z, 0, 2^b - 1);
// 0 for a non-finite group.
template <int BITS>
__device__ __forceinline__ uint32_t group_encode(float x, const GroupParams& gp) {
  constexpr int QMAX = (1 << BITS) - 1;
  if (!gp.finite) return 0u;
  const float tq = rintf(__fdiv_rn(x, gp.sf)) + gp.zf;
  return (uint32_t)fminf(fmaxf(tq, 0.f), (float)QMAX);
}

// One lane's share of a group: 8 channels.
struct Quant8 {
  uint32_t w0, w1;  // packed codes: INT2 -> w0 (2 bytes), INT4 -> w0 (4 bytes), INT8 -> w0, w1
  __half s, z;      // the group's scale and zero-point
  uint32_t flags;   // KVQ_FLAG_ZERO_CLAMPED / KVQ_FLAG_NONFINITE
};

// Quantizes 8 channels held by this lane; the group is the `tpg` adjacent
// lanes (tpg = g / 8, a power of two <= 32, groups aligned to tpg lanes).
// Every lane of the warp must call it (the group min/max uses shuffles).
//
// SYM selects the symmetric (absmax) grid: the zero-centred grid that "What
// actually happens when you quantize a KV cache", section 3, compares the
// asymmetric one against, written out as the absmax quantizer in "Serving
// many users at once", "Quantization: rounding the weights":
//   a = max |x|, s = the smallest fp16 with s * (2^(b-1) - 1) >= a
//   (s = 1 when a = 0), q = clamp(rint(x / s), -2^(b-1), 2^(b-1) - 1),
//   stored as the code q + 2^(b-1); z is returned as 2^(b-1) and not stored.
template <int BITS, bool SYM = false>
__device__ __forceinline__ Quant8 quantize8(const uint4 v, int tpg) {
  constexpr int HALF = 1 << (BITS - 1);  // symmetric code offset
  const __half* h = reinterpret_cast<const __half*>(&v);
  float mn = INFINITY, mx = -INFINITY;
  bool finite = true;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float f = __half2float(h[k]);
    finite = finite && isfinite(f);
    mn = fminf(mn, f);
    mx = fmaxf(mx, f);
  }
  for (int o = 1; o < tpg; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    finite = (__shfl_xor_sync(0xffffffffu, (int)finite, o) != 0) && finite;
  }

  Quant8 r;
  r.s = __ushort_as_half(0);
  r.z = __ushort_as_half(0);
  r.flags = 0;
  r.w0 = 0;
  r.w1 = 0;
  if constexpr (SYM) {
    r.z = __int2half_rn(HALF);
    float sf = 0.f;
    if (!finite) {
      r.flags |= KVQ_FLAG_NONFINITE;
    } else {
      const float a = fmaxf(fabsf(mn), fabsf(mx));
      r.s = (a == 0.f) ? __float2half_rn(1.f) : quant_detail::scale_round_up((double)a, HALF - 1);
      sf = __half2float(r.s);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float t = 0.f;
      if (finite) t = fminf(fmaxf(rintf(__fdiv_rn(__half2float(h[k]), sf)), (float)-HALF), (float)(HALF - 1));
      const uint32_t q = (uint32_t)(int)(t + (float)HALF);
      if constexpr (BITS == 2) {
        r.w0 |= q << (2 * k);
      } else if constexpr (BITS == 4) {
        r.w0 |= q << (4 * k);
      } else {
        if (k < 4) r.w0 |= q << (8 * k);
        else       r.w1 |= q << (8 * (k - 4));
      }
    }
    return r;
  }
  const GroupParams gp = group_params<BITS>(mn, mx, finite);
  r.s = gp.s;
  r.z = gp.z;
  r.flags = gp.flags;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t q = group_encode<BITS>(__half2float(h[k]), gp);
    if constexpr (BITS == 2) {
      r.w0 |= q << (2 * k);  // channel 4m + j -> bits 2j of byte m
    } else if constexpr (BITS == 4) {
      r.w0 |= q << (4 * k);  // channel 2m -> low nibble of byte m
    } else {
      if (k < 4) r.w0 |= q << (8 * k);
      else       r.w1 |= q << (8 * (k - 4));
    }
  }
  return r;
}

// NF4 ("Gör inference billig", NF4: sixteen normal-quantile levels with a
// block absmax scale).  s = max |x| over the group (an fp16 value, exact);
// code = number of level midpoints (`mid`, fp32, increasing) below x/s, i.e.
// the nearest level with ties to the lower one; a group of zeros or with
// inf/NaN stores s = 0 and codes 0 (the latter flagged).  Same lane layout
// and packing as quantize8<4>.
__device__ __forceinline__ Quant8 quantize8_nf4(const uint4 v, int tpg, const float (&mid)[16]) {
  const __half* h = reinterpret_cast<const __half*>(&v);
  float a = 0.f;
  bool finite = true;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float f = __half2float(h[k]);
    finite = finite && isfinite(f);
    a = fmaxf(a, fabsf(f));
  }
  for (int o = 1; o < tpg; o <<= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    finite = (__shfl_xor_sync(0xffffffffu, (int)finite, o) != 0) && finite;
  }
  Quant8 r;
  r.flags = finite ? 0u : KVQ_FLAG_NONFINITE;
  const bool live = finite && a > 0.f;
  r.s = live ? __float2half_rn(a) : __ushort_as_half(0);
  r.z = __ushort_as_half(0);
  r.w0 = 0;
  r.w1 = 0;
  if (live) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float t = __fdiv_rn(__half2float(h[k]), a);
      uint32_t q = 0;
#pragma unroll
      for (int i = 0; i < 15; ++i) q += (mid[i] < t) ? 1u : 0u;
      r.w0 |= q << (4 * k);
    }
  }
  return r;
}

}  // namespace kvq
