// Quantize-on-append kernel.
//
// One thread owns one group of `g` consecutive channels of one new K or V
// vector ("What actually happens when you quantize a KV cache", section 3
// steps 2-5 and section 4): it scans the group for min and max, derives the
// fp16 scale and the integer zero-point, encodes every channel and packs two
// INT4 codes per byte with the even channel in the low nibble.  Consecutive
// threads own consecutive groups of the same vector, so the fp16 reads, the
// code writes and the header writes are all contiguous across a warp.
//
// Arithmetic (fixed so that codes are reproducible bit for bit):
//   range = max - min            fp64 (exact for two fp16 values)
//   s     = fp16 rounded toward +inf of range / (2^b - 1), fp64 quotient
//   z     = rint(-min / s)       fp32 IEEE division, round half to even
//   q     = clamp(rint(x / s) + z, 0, 2^b - 1)
// The file is compiled without fast-math: '/' here must stay div.rn.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

__device__ __forceinline__ __half half_round_up(double d) {
  unsigned short h;
  asm("cvt.rp.f16.f64 %0, %1;" : "=h"(h) : "d"(d));
  return __ushort_as_half(h);
}

template <int BITS>
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const CacheGeom& c = p.geom;
  const int which = blockIdx.y;  // 0: K, 1: V
  const int units_per_row = (BITS == 16) ? c.D / 8 : c.ngroups;
  const long long n_units = (long long)p.batch * p.num_new * c.Hkv * units_per_row;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n_units) return;

  const int grp = (int)(u % units_per_row);
  long long r = u / units_per_row;
  const int kvh = (int)(r % c.Hkv);
  r /= c.Hkv;
  const int t = (int)(r % p.num_new);
  const int b = (int)(r / p.num_new);

  uint32_t flags = 0;
  const int pos = __ldg(p.seq_lens_before + b) + t;
  const int limit = (c.layout == KVQ_DENSE) ? c.slots : c.max_blocks * c.slots;
  long long row = -1;
  if (pos < 0 || pos >= limit) {
    flags |= KVQ_FLAG_SEQ_LEN;
  } else {
    row = token_row(c, b, kvh, pos);
    if (row < 0) flags |= KVQ_FLAG_BLOCK_TABLE;
  }
  if (row < 0) {
    if (p.status) atomicOr(p.status, flags);
    return;
  }

  const __half* src = p.src[which] + (((long long)b * p.num_new + t) * c.Hkv + kvh) * c.D;

  if constexpr (BITS == 16) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + grp);
    *reinterpret_cast<uint4*>(p.codes[which] + row * c.row_bytes + grp * 16) = v;
    return;
  } else {
    constexpr int QMAX = (1 << BITS) - 1;
    const int g = c.g;
    const uint4* gsrc = reinterpret_cast<const uint4*>(src + (long long)grp * g);

    // pass 1: min, max, finiteness
    float mn = INFINITY, mx = -INFINITY;
    bool finite = true;
    for (int i = 0; i < g / 8; ++i) {
      const uint4 v = __ldg(gsrc + i);
      const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(h2[k]);
        finite = finite && isfinite(f.x) && isfinite(f.y);
        mn = fminf(mn, fminf(f.x, f.y));
        mx = fmaxf(mx, fmaxf(f.x, f.y));
      }
    }

    __half s_h = __ushort_as_half(0);
    __half z_h = __ushort_as_half(0);
    float sf = 0.f, zf = 0.f;
    if (!finite) {
      flags |= KVQ_FLAG_NONFINITE;
    } else {
      const double range = (double)mx - (double)mn;
      if (range == 0.0) {
        // constant group: s = |min| (1 for an all-zero group) decodes exactly
        s_h = __float2half_rn(mn == 0.f ? 1.f : fabsf(mn));
      } else {
        s_h = half_round_up(range / (double)QMAX);
      }
      sf = __half2float(s_h);
      zf = rintf(__fdiv_rn(-mn, sf));
      if (fabsf(zf) > 2048.f) {
        flags |= KVQ_FLAG_ZERO_CLAMPED;
        zf = fminf(fmaxf(zf, -2048.f), 2048.f);
      }
      z_h = __int2half_rn((int)zf);  // an integer of magnitude <= 2048: exact, +0 for 0
    }

    // pass 2: encode and pack, 8 channels (one 16-byte load) at a time
    uint8_t* dst = p.codes[which] + row * c.row_bytes + (long long)grp * g * BITS / 8;
    for (int i = 0; i < g / 8; ++i) {
      const uint4 v = __ldg(gsrc + i);
      const __half* h = reinterpret_cast<const __half*>(&v);
      uint32_t w0 = 0, w1 = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t q = 0;
        if (finite) {
          const float tq = rintf(__fdiv_rn(__half2float(h[k]), sf)) + zf;
          q = (uint32_t)fminf(fmaxf(tq, 0.f), (float)QMAX);
        }
        if constexpr (BITS == 4) {
          w0 |= q << (4 * k);  // channel 2m -> low nibble of byte m
        } else {
          if (k < 4) w0 |= q << (8 * k);
          else       w1 |= q << (8 * (k - 4));
        }
      }
      if constexpr (BITS == 4) {
        *reinterpret_cast<uint32_t*>(dst + i * 4) = w0;
      } else {
        *reinterpret_cast<uint2*>(dst + i * 8) = make_uint2(w0, w1);
      }
    }
    const long long h_idx = row * c.ngroups + grp;
    p.scale[which][h_idx] = s_h;
    p.zero[which][h_idx] = z_h;
    if (flags && p.status) atomicOr(p.status, flags);
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const CacheGeom& c = p.geom;
  const int units_per_row = (c.bits == 16) ? c.D / 8 : c.ngroups;
  const long long n_units = (long long)p.batch * p.num_new * c.Hkv * units_per_row;
  if (n_units == 0) return cudaSuccess;
  const dim3 block(256);
  const dim3 grid((unsigned)((n_units + 255) / 256), 2);
  switch (c.bits) {
    case 4:  append_kernel<4><<<grid, block, 0, stream>>>(p); break;
    case 8:  append_kernel<8><<<grid, block, 0, stream>>>(p); break;
    default: append_kernel<16><<<grid, block, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace kvq
