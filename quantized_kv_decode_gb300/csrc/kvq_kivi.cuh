// Axis-aware (KIVI-style) one-token append, shared by the append kernel and
// the tensor-core decode kernel's fused step.
//
// "What actually happens when you quantize a KV cache", section 3 step 7
// ("axis choice": a K group is one channel across consecutive tokens; V
// keeps per-token groups; the tokens of a block that has not filled yet
// stay in an fp16 residual window; "sinks": the first tokens stay fp16) and
// section 7.  The quantizer is the asymmetric one of section 3 steps 2-5
// and section 4 (group_params / group_encode / quantize8), so a K group is
// exactly a per-token group with its axis turned.
#pragma once

#include "kvq_quant.cuh"

namespace kvq {

// Where an axis-aware append reads and writes.  src: the new tokens
// [batch][num_new][Hkv][D] fp16 (K, V); window: the fp16 sinks and residual
// ring [batch][Hkv][sink + g][D] (K, V); codes / scale / zero: the cache
// arrays (K: per-channel headers [..][D] per block; V: per-token headers).
struct KiviIO {
  const CacheGeom* geom;
  uint8_t* codes[2];
  __half* scale[2];
  __half* zero[2];
  const __half* src[2];
  __half* window[2];
  uint32_t* status;
  int num_new;
};

// fp16 source of token q of sequence b, KV head kvh: the residual window for
// tokens cached before this append (p0 = the length before it), the new
// input otherwise
__device__ __forceinline__ const __half* kivi_token_src(const KiviIO& io, int which, int b,
                                                        int kvh, int q, int p0) {
  const CacheGeom& c = *io.geom;
  if (q < p0) {
    const long long bh = (long long)b * c.Hkv + kvh;
    return io.window[which] + (bh * (c.sink + c.g) + c.sink + (q - c.sink) % c.g) * c.D;
  }
  return io.src[which] + (((long long)b * io.num_new + (q - p0)) * c.Hkv + kvh) * c.D;
}

// The caller array kivi_token_src reads for token q (debug-build checks).
__device__ __forceinline__ int kivi_src_array(int which, int q, int p0) {
  return q < p0 ? (which ? KVQ_ARRAY_V_WINDOW : KVQ_ARRAY_K_WINDOW)
                : (which ? KVQ_ARRAY_V_NEW : KVQ_ARRAY_K_NEW);
}

// Quantizes block j (positions [start, start + g)) of sequence b, KV head
// kvh, whose tokens before p0 sit in the residual window and the rest in the
// new input.  Every thread of the CTA calls it (any whole number of warps).
template <int BITS>
__device__ void kivi_quantize_block(const KiviIO& io, int b, int kvh, int j, long long start,
                                    int p0) {
  const CacheGeom& c = *io.geom;
  const int g = c.g, D = c.D;
  uint32_t flags = 0;
  const long long hrow = kch_hdr(c, b, kvh, j);  // the block's K header row (x D)

  // ---- K: one group per channel over the block's g tokens ----
  constexpr int CPU = BITS == 4 ? 2 : 1;  // channels per code byte
  for (int u = threadIdx.x; u < D / CPU; u += blockDim.x) {
    GroupParams gp[CPU];
#pragma unroll
    for (int e = 0; e < CPU; ++e) {
      const int ch = u * CPU + e;
      float mn = INFINITY, mx = -INFINITY;
      bool finite = true;
      for (int t = 0; t < g; ++t) {
        const __half* xp = kivi_token_src(io, 0, b, kvh, (int)start + t, p0) + ch;
        const float x = KVQ_IN(c, kivi_src_array(0, (int)start + t, p0), xp, 2) ? __half2float(*xp)
                                                                               : 0.f;
        finite = finite && isfinite(x);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
      gp[e] = group_params<BITS>(mn, mx, finite);
      flags |= gp[e].flags;
      if (hrow >= 0) {
        if (KVQ_IN(c, KVQ_ARRAY_K_SCALE, io.scale[0] + hrow * D + ch, 2))
          io.scale[0][hrow * D + ch] = gp[e].s;
        if (KVQ_IN(c, KVQ_ARRAY_K_ZERO, io.zero[0] + hrow * D + ch, 2))
          io.zero[0][hrow * D + ch] = gp[e].z;
      } else {
        flags |= KVQ_FLAG_BLOCK_TABLE;
      }
    }
    for (int t = 0; t < g; ++t) {
      const __half* src = kivi_token_src(io, 0, b, kvh, (int)start + t, p0) + u * CPU;
      const bool src_ok = KVQ_IN(c, kivi_src_array(0, (int)start + t, p0), src, 2 * CPU);
      uint32_t byte = 0;
#pragma unroll
      for (int e = 0; e < CPU; ++e)
        byte |= group_encode<BITS>(src_ok ? __half2float(src[e]) : 0.f, gp[e]) << (4 * e);
      const long long row = kch_row(c, b, kvh, (int)start + t);
      if (row < 0) flags |= KVQ_FLAG_BLOCK_TABLE;
      else if (KVQ_IN(c, KVQ_ARRAY_K_CODES, io.codes[0] + row * c.row_bytes + u, 1))
        io.codes[0][row * c.row_bytes + u] = (uint8_t)byte;
    }
  }

  // ---- V: per-token groups of g channels (quantize8 over 8-channel chunks) ----
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chv = D / 8;               // chunks per token
  const int tpw = 32 / chv;            // tokens per warp pass (D <= 256)
  const int tpg = g / 8;               // lanes per group
  for (int t0 = warp * tpw; t0 < g; t0 += (blockDim.x / 32) * tpw) {
    const int t = t0 + lane / chv, ch = lane % chv;  // every lane is live: g % tpw == 0
    const long long q = start + t;
    const uint4* vp = reinterpret_cast<const uint4*>(kivi_token_src(io, 1, b, kvh, (int)q, p0)) + ch;
    const uint4 v = KVQ_IN(c, kivi_src_array(1, (int)q, p0), vp, 16) ? *vp : make_uint4(0u, 0u, 0u, 0u);
    const Quant8 qz = quantize8<BITS>(v, tpg);
    const long long row = kch_row(c, b, kvh, (int)q);
    if (row < 0) {
      flags |= KVQ_FLAG_BLOCK_TABLE;
      continue;
    }
    uint8_t* dst = io.codes[1] + row * c.row_bytes + ch * BITS;
    if (KVQ_IN(c, KVQ_ARRAY_V_CODES, dst, BITS)) {
      if constexpr (BITS == 4) {
        *reinterpret_cast<uint32_t*>(dst) = qz.w0;
      } else {
        *reinterpret_cast<uint2*>(dst) = make_uint2(qz.w0, qz.w1);
      }
    }
    if (ch % tpg == 0) {
      const long long hi = row * c.ngroups + ch / tpg;
      if (KVQ_IN(c, KVQ_ARRAY_V_SCALE, io.scale[1] + hi, 2)) io.scale[1][hi] = qz.s;
      if (KVQ_IN(c, KVQ_ARRAY_V_ZERO, io.zero[1] + hi, 2)) io.zero[1][hi] = qz.z;
      flags |= qz.flags;
    }
  }
  if (flags && io.status) atomicOr(io.status, flags);
}

// The one-token append of sequence b, KV head kvh (p0 tokens cached before
// it, io.num_new == 1): the token either completes its block, which is then
// quantized (window rows read), or goes to its fp16 slot (a sink or the
// residual ring).  Every thread of the CTA calls it; a position beyond the
// cache flags KVQ_FLAG_SEQ_LEN (once per sequence) and writes nothing.
template <int BITS>
__device__ void kivi_append_one(const KiviIO& io, int b, int kvh, int p0) {
  const CacheGeom& c = *io.geom;
  if (p0 < 0 || p0 >= kch_capacity(c)) {
    if (threadIdx.x == 0 && kvh == 0 && io.status) atomicOr(io.status, KVQ_FLAG_SEQ_LEN);
    return;
  }
  const int slot = window_slot(c, p0 + 1, p0);
  if (slot < 0) {  // p0 ends its block
    const int j = (p0 - c.sink) / c.g;
    kivi_quantize_block<BITS>(io, b, kvh, j, (long long)c.sink + (long long)j * c.g, p0);
    return;
  }
  const long long bh = (long long)b * c.Hkv + kvh;
  const int chunks = c.D / 8;
  if (threadIdx.x < 2 * chunks) {
    const int which = threadIdx.x / chunks, ch = threadIdx.x % chunks;
    uint4* to = reinterpret_cast<uint4*>(io.window[which] + (bh * (c.sink + c.g) + slot) * c.D) + ch;
    const uint4* from = reinterpret_cast<const uint4*>(io.src[which] + bh * c.D) + ch;
    if (KVQ_IN(c, which ? KVQ_ARRAY_V_NEW : KVQ_ARRAY_K_NEW, from, 16) &&
        KVQ_IN(c, which ? KVQ_ARRAY_V_WINDOW : KVQ_ARRAY_K_WINDOW, to, 16))
      *to = *from;
  }
}

}  // namespace kvq
