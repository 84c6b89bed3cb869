// Quantize-on-append kernel.
//
// Each group of `g` consecutive channels of one new K or V vector is encoded
// by quantize8() (kvq_quant.cuh; "What actually happens when you quantize a
// KV cache", section 3 steps 2-5 and section 4).  One thread owns 8 channels
// (one 16-byte load); the g/8 threads of a group are adjacent lanes of one
// warp and combine their min/max with shuffles, so every lane runs a short
// chain (this matters most for the one-token append of a decode step).
// Reads, code writes and header writes are contiguous across a warp.
#include "kvq_quant.cuh"

namespace kvq {
namespace {

// KIND: 0 asymmetric, 1 symmetric, 2 NF4 (BITS 4)
template <int BITS, int KIND>
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr bool SYM = KIND == 1;
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
  const int32_t* lp = p.seq_lens_before + b;
  const int pos = KVQ_IN(c, KVQ_ARRAY_SEQ_LENS, lp, 4) ? __ldg(lp) + t : -1;
  const int limit = (c.layout == KVQ_DENSE) ? c.slots : c.max_blocks * c.slots;
  long long row = -1;
  if (pos < 0 || pos >= limit) {
    flags |= KVQ_FLAG_SEQ_LEN;
  } else {
    row = token_row(c, b, kvh, pos);
    if (row < 0) flags |= KVQ_FLAG_BLOCK_TABLE;
  }
  const __half* src = p.src[which] + (((long long)b * p.num_new + t) * c.Hkv + kvh) * c.D;
  const int a_src = which ? KVQ_ARRAY_V_NEW : KVQ_ARRAY_K_NEW;
  const int a_codes = which ? KVQ_ARRAY_V_CODES : KVQ_ARRAY_K_CODES;

  if constexpr (BITS == 16) {
    if (!live) return;
    if (row < 0) {
      if (ch == 0 && p.status) atomicOr(p.status, flags);
      return;
    }
    const uint4* sp = reinterpret_cast<const uint4*>(src) + ch;
    const uint4 v = KVQ_IN(c, a_src, sp, 16) ? __ldg(sp) : make_uint4(0u, 0u, 0u, 0u);
    uint8_t* dst = p.codes[which] + row * c.row_bytes + ch * 16;
    if (KVQ_IN(c, a_codes, dst, 16)) *reinterpret_cast<uint4*>(dst) = v;
    return;
  } else {
    const int tpg = c.g / 8;          // threads per group: 1, 2, 4, ..., 32
    const int sub = ch % tpg;          // this thread's place in its group
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (live && KVQ_IN(c, a_src, reinterpret_cast<const uint4*>(src) + ch, 16))
      v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
    // every lane: the group uses shuffles
    const Quant8 qz = KIND == 2 ? quantize8_nf4(v, tpg, p.nf4_mid) : quantize8<BITS, SYM>(v, tpg);
    if (!live) return;
    if (row < 0) {
      if (ch == 0 && p.status) atomicOr(p.status, flags);
      return;
    }
    flags |= qz.flags;
    const uint32_t w0 = qz.w0, w1 = qz.w1;
    const __half s_h = qz.s, z_h = qz.z;
    uint8_t* dst = p.codes[which] + row * c.row_bytes + (long long)ch * 8 * BITS / 8;
    if (KVQ_IN(c, a_codes, dst, BITS)) {
      if constexpr (BITS == 2) {
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w0;
      } else if constexpr (BITS == 4) {
        *reinterpret_cast<uint32_t*>(dst) = w0;
      } else {
        *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
      }
    }
    if (sub == 0) {
      const long long h_idx = row * c.ngroups + ch / tpg;
      if (KVQ_IN(c, which ? KVQ_ARRAY_V_SCALE : KVQ_ARRAY_K_SCALE, p.scale[which] + h_idx, 2))
        p.scale[which][h_idx] = s_h;
      if constexpr (KIND == 0)
        if (KVQ_IN(c, which ? KVQ_ARRAY_V_ZERO : KVQ_ARRAY_K_ZERO, p.zero[which] + h_idx, 2))
          p.zero[which][h_idx] = z_h;
      if (flags && p.status) atomicOr(p.status, flags);
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const CacheGeom& c = p.geom;
  if (c.kch) return launch_append_kivi(p, stream);
  const long long n_units = (long long)p.batch * p.num_new * c.Hkv * (c.D / 8);
  if (n_units == 0) return cudaSuccess;
  const dim3 block(256);
  const dim3 grid((unsigned)((n_units + 255) / 256), 2);
  const int kind = c.nf4 ? 2 : (c.sym ? 1 : 0);
  switch (c.bits * 4 + kind) {
    case 8:  return launch_pdl(append_kernel<2, 0>, grid, block, 0, stream, p);
    case 9:  return launch_pdl(append_kernel<2, 1>, grid, block, 0, stream, p);
    case 16: return launch_pdl(append_kernel<4, 0>, grid, block, 0, stream, p);
    case 17: return launch_pdl(append_kernel<4, 1>, grid, block, 0, stream, p);
    case 18: return launch_pdl(append_kernel<4, 2>, grid, block, 0, stream, p);
    case 32: return launch_pdl(append_kernel<8, 0>, grid, block, 0, stream, p);
    case 33: return launch_pdl(append_kernel<8, 1>, grid, block, 0, stream, p);
    default: return launch_pdl(append_kernel<16, 0>, grid, block, 0, stream, p);
  }
}

}  // namespace kvq
