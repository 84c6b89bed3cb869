// Quantize-on-append kernel.
//
// Each group of `g` consecutive channels of one new K or V vector is encoded
// as in "What actually happens when you quantize a KV cache" (section 3 steps
// 2-5 and section 4): min and max over the group, an fp16 scale and integer
// zero-point, codes clamp(round(x/s) + z, 0, 2^b - 1), and two INT4 codes per
// byte with the even channel in the low nibble.
//
// One thread owns 8 channels (one 16-byte load); the g/8 threads of a group
// are adjacent lanes of one warp and combine their min/max with shuffles, so
// every lane runs a short chain (this matters most for the one-token append
// of a decode step, where there are few groups).  Reads, code writes and
// header writes are contiguous across a warp.
//
// Arithmetic (fixed so that codes are reproducible bit for bit):
//   range = max - min            fp64 (exact for two fp16 values)
//   s     = the smallest fp16 with s * (2^b - 1) >= range (range / (2^b - 1)
//           rounded toward +inf): an fp32 estimate, then exact fp64 checks
//   z     = rint(-min / s)       fp32 IEEE division, round half to even
//   q     = clamp(rint(x / s) + z, 0, 2^b - 1)
// The file is compiled without fast-math: '/' here must stay div.rn.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

__device__ __forceinline__ unsigned short half_bits_up(unsigned short h) {   // h >= 0 finite
  return (unsigned short)(h + 1);
}
__device__ __forceinline__ unsigned short half_bits_down(unsigned short h) { // h > 0
  return (unsigned short)(h - 1);
}
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
  if (half_bits_value(h) * qmax < range) h = half_bits_up(h);
  if (h > 1 && half_bits_value(half_bits_down(h)) * qmax >= range) h = half_bits_down(h);
  return __ushort_as_half(h);
}

template <int BITS>
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const CacheGeom& c = p.geom;
  const int which = blockIdx.y;  // 0: K, 1: V
  const int chunks = c.D / 8;    // 8-channel chunks per vector
  const long long n_units = (long long)p.batch * p.num_new * c.Hkv * chunks;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = u < n_units;
  const long long uu = live ? u : 0;

  const int ch = (int)(uu % chunks);
  long long r = uu / chunks;
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
  const __half* src = p.src[which] + (((long long)b * p.num_new + t) * c.Hkv + kvh) * c.D;

  if constexpr (BITS == 16) {
    if (!live) return;
    if (row < 0) {
      if (ch == 0 && p.status) atomicOr(p.status, flags);
      return;
    }
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
    *reinterpret_cast<uint4*>(p.codes[which] + row * c.row_bytes + ch * 16) = v;
    return;
  } else {
    constexpr int QMAX = (1 << BITS) - 1;
    const int tpg = c.g / 8;          // threads per group: 1, 2, 4, ..., 32
    const int sub = ch % tpg;          // this thread's place in its group
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (live) v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
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
    // combine over the group's adjacent lanes (groups never straddle a warp)
    for (int o = 1; o < tpg; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      finite = (__shfl_xor_sync(0xffffffffu, (int)finite, o) != 0) && finite;
    }
    if (!live) return;
    if (row < 0) {
      if (ch == 0 && p.status) atomicOr(p.status, flags);
      return;
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
        s_h = scale_round_up(range, QMAX);
      }
      sf = __half2float(s_h);
      zf = rintf(__fdiv_rn(-mn, sf));
      if (fabsf(zf) > 2048.f) {
        flags |= KVQ_FLAG_ZERO_CLAMPED;
        zf = fminf(fmaxf(zf, -2048.f), 2048.f);
      }
      z_h = __int2half_rn((int)zf);  // an integer of magnitude <= 2048: exact, +0 for 0
    }

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
    uint8_t* dst = p.codes[which] + row * c.row_bytes + (long long)ch * 8 * BITS / 8;
    if constexpr (BITS == 4) {
      *reinterpret_cast<uint32_t*>(dst) = w0;
    } else {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
    }
    if (sub == 0) {
      const long long h_idx = row * c.ngroups + ch / tpg;
      p.scale[which][h_idx] = s_h;
      p.zero[which][h_idx] = z_h;
      if (flags && p.status) atomicOr(p.status, flags);
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const CacheGeom& c = p.geom;
  const long long n_units = (long long)p.batch * p.num_new * c.Hkv * (c.D / 8);
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
