// CUDA-core split-K decode attention for the shapes the tensor-core kernels
// do not take: head_dim 256, more than 8 query heads per KV head (fp16
// caches included), INT4 / NF4 with groups of 8/16 channels or one group per
// head, INT2 at head_dim 64 or with more (group, head) columns than one
// V-mma n-tile.
//
// What it computes is the decode step of "Quantization & inference
// optimisation" ("Prefill, then decode": scores = K q / sqrt(d), softmax,
// weighted V over every cached row), reading the codes and dequantizing them
// in registers ("What actually happens when you quantize a KV cache",
// sections 3-4 and 6; NF4 codes index the normal-quantile levels of "Gör
// inference billig").
//
// One CTA per (split, KV head, sequence), 4 warps; each warp streams its own
// 32-token tiles with no block-wide barrier until the end:
//  * scores, lane = token: the lane reads its token's code row with 16-byte
//    loads, converts each code, and accumulates q . code per group for every
//    query head (q from shared memory, read by all lanes at once); per group
//    the scale and zero-point enter once: s (sum q c - z sum q).
//  * online softmax per head (warp max, log2 domain); the probabilities go to
//    shared memory.
//  * weighted V, lane = 32-th of the channels: per token of the tile the lane
//    dequantizes its channels and accumulates p * v_hat for every head.
//  * the warps' (m, l, o) are merged in shared memory; the CTA writes the
//    final row (one split) or its partial for the merge kernel.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {
namespace cc {

constexpr int kWarps = 4;
constexpr int kTok = 32;  // tokens per warp tile

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// code k (0-based) of a 16-byte chunk holding 128 / BITS codes (little-endian
// bit order: INT4 even channel in the low nibble, INT2 channel 4m + j in bits
// 2j of byte m)
template <int BITS>
__device__ __forceinline__ uint32_t code_of(const uint4& w, int k) {
  const uint32_t word = k < 32 / BITS * 1 ? w.x : (k < 2 * 32 / BITS ? w.y : (k < 3 * 32 / BITS ? w.z : w.w));
  const int kk = k % (32 / BITS);
  return (word >> (BITS * kk)) & ((1u << BITS) - 1u);
}

template <int BITS, int D, int GP>
struct CcCfg {
  static constexpr int ROWB = D * BITS / 8;  // bytes per row
  static constexpr int NCH = ROWB / 16;      // 16-byte chunks per row
  static constexpr int EPC = 128 / BITS;     // codes (channels) per chunk
  static constexpr int CPL = D / 32;         // V channels per lane
  static_assert(ROWB % 16 == 0, "row of 16-byte chunks");
};

template <int BITS, int D, int GP>
size_t cc_smem_bytes() {
  // q [GP][D], per-group sums of q [GP][D/8], probabilities [warps][tok][GP],
  // NF4 levels [16], merge [warps][GP][D] + [warps][GP][2]
  return sizeof(float) * ((size_t)GP * D + GP * (D / 8) + kWarps * kTok * GP + 16 +
                          kWarps * GP * (D + 2));
}

template <int BITS, int D, int GP>
__global__ void __launch_bounds__(kWarps * 32) decode_cc_kernel(const DecodeParams p) {
  using C = CcCfg<BITS, D, GP>;
  extern __shared__ __align__(16) float smem[];
  const CacheGeom& c = p.geom;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  float* q_s = smem;                          // [GP][D]
  float* qg_s = q_s + GP * D;                 // [GP][groups] sum of q over each group
  float* p_s = qg_s + GP * (D / 8);           // [warps][kTok][GP]
  float* lv_s = p_s + kWarps * kTok * GP;     // [16] NF4 levels
  float* red = lv_s + 16;                     // [warps][GP][D]
  float* ml = red + kWarps * GP * D;          // [warps][GP][2]

  int L = seq_len_of(p, b);
  if (L < 0 || L > p.len_limit) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0 && p.status) atomicOr(p.status, KVQ_FLAG_SEQ_LEN);
    L = 0;
  }
  const int t0 = split * p.chunk;
  const int t1 = min(L, t0 + p.chunk);
  if (p.splits > 1 && t0 >= L) return;  // the merge reads splits < ceil(L / chunk) only

  const __half* qg = p.q + ((long long)b * p.Hq + (long long)kvh * G) * D;
  for (int i = threadIdx.x; i < GP * D; i += kWarps * 32)
    q_s[i] = (i < G * D && KVQ_IN(c, KVQ_ARRAY_Q, qg + i, 2)) ? __half2float(qg[i]) : 0.f;
  if (threadIdx.x < 16) lv_s[threadIdx.x] = c.nf4 ? p.nf4_level[threadIdx.x] : 0.f;
  __syncthreads();

  const int gsz = BITS == 16 ? D : c.g;    // channels per group
  const int ngr = BITS == 16 ? 1 : c.ngroups;
  for (int i = threadIdx.x; i < GP * ngr; i += kWarps * 32) {
    const int h = i / ngr, g = i - h * ngr;
    float sum = 0.f;
    for (int d = g * gsz; d < (g + 1) * gsz; ++d) sum += q_s[h * D + d];
    qg_s[h * ngr + g] = sum;
  }
  __syncthreads();
  const bool sym = c.sym != 0, nf4 = c.nf4 != 0;
  const float zsym = (float)(1 << (BITS == 16 ? 0 : BITS - 1));

  float m_run[GP], l_lane[GP], o[GP][C::CPL];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    m_run[h] = -INFINITY;
    l_lane[h] = 0.f;
#pragma unroll
    for (int e = 0; e < C::CPL; ++e) o[h][e] = 0.f;
  }
  bool bt_bad = false;
  float* pw = p_s + warp * kTok * GP;
  const int ntiles = t1 > t0 ? (t1 - t0 + kTok - 1) / kTok : 0;

  for (int it = warp; it < ntiles; it += kWarps) {
    const int ts = t0 + it * kTok;
    const int tok = ts + lane;
    long long row = -1;
    if (tok < t1) {
      row = token_row(c, b, kvh, tok);
      bt_bad |= row < 0;
    }

    // ---- scores: this lane's token ----
    float sc[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) sc[h] = 0.f;
    if (row >= 0) {
      const uint4* kr = reinterpret_cast<const uint4*>(p.codes[0] + row * C::ROWB);
      const bool k_ok = KVQ_IN(c, KVQ_ARRAY_K_CODES, kr, C::ROWB);
      if constexpr (BITS == 16) {
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          const uint4 w = k_ok ? __ldg(kr + ch) : make_uint4(0u, 0u, 0u, 0u);
          const __half* hv = reinterpret_cast<const __half*>(&w);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float x = __half2float(hv[e]);
            const int d = ch * 8 + e;
#pragma unroll
            for (int h = 0; h < GP; ++h) sc[h] = fmaf(q_s[h * D + d], x, sc[h]);
          }
        }
      } else {
        // per group: s * (sum q c - z sum q), or for NF4 s * sum q level(c);
        // groups are a power of two >= 8 channels, so a group can only end
        // at a channel index that is a multiple of 8
        float acc[GP];
        int gcur = 0;
#pragma unroll
        for (int h = 0; h < GP; ++h) acc[h] = 0.f;
        auto flush = [&]() {
          const long long hi = row * ngr + gcur;
          const float s = KVQ_IN(c, KVQ_ARRAY_K_SCALE, p.scale[0] + hi, 2) ? __half2float(p.scale[0][hi]) : 0.f;
          const float z = nf4 ? 0.f
                        : (sym ? zsym
                               : (KVQ_IN(c, KVQ_ARRAY_K_ZERO, p.zero[0] + hi, 2) ? __half2float(p.zero[0][hi])
                                                                                 : 0.f));
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            sc[h] = fmaf(s, fmaf(-z, qg_s[h * ngr + gcur], acc[h]), sc[h]);
            acc[h] = 0.f;
          }
          ++gcur;
        };
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          const uint4 w = k_ok ? __ldg(kr + ch) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int e = 0; e < C::EPC; ++e) {
            const int d = ch * C::EPC + e;
            if ((d & 7) == 0 && d > 0 && (d & (gsz - 1)) == 0) flush();
            const uint32_t q = code_of<BITS>(w, e);
            const float x = nf4 ? lv_s[q] : (float)q;
#pragma unroll
            for (int h = 0; h < GP; ++h) acc[h] = fmaf(q_s[h * D + d], x, acc[h]);
          }
        }
        flush();
      }
    }
#pragma unroll
    for (int h = 0; h < GP; ++h) sc[h] = (row >= 0 && h < G) ? sc[h] * p.scale_log2 : -INFINITY;

    // ---- online softmax per head over the tile ----
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      float mt = sc[h];
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o2));
      const float mn = fmaxf(m_run[h], mt);
      const float alpha = (m_run[h] == -INFINITY) ? (mn == -INFINITY ? 1.f : 0.f) : ex2(m_run[h] - mn);
      const float pv = (sc[h] == -INFINITY) ? 0.f : ex2(sc[h] - mn);
      l_lane[h] = fmaf(l_lane[h], alpha, pv);
#pragma unroll
      for (int e = 0; e < C::CPL; ++e) o[h][e] *= alpha;
      m_run[h] = mn;
      pw[lane * GP + h] = pv;
    }
    __syncwarp();

    // ---- weighted V: this lane's channels ----
    const int d0 = lane * C::CPL;
    const int gv = d0 / gsz;  // the lane's channels lie in one group (gsz >= 8 >= CPL)
    const int nt = min(kTok, t1 - ts);
    for (int t = 0; t < nt; ++t) {
      const long long vr = __shfl_sync(0xffffffffu, row, t);
      if (vr < 0) continue;  // warp-uniform
      float x[C::CPL];
      const uint8_t* rp = p.codes[1] + vr * C::ROWB;
      const bool v_ok = KVQ_IN(c, KVQ_ARRAY_V_CODES, rp, C::ROWB);
      if constexpr (BITS == 16) {
        const __half* hv = reinterpret_cast<const __half*>(rp) + d0;
#pragma unroll
        for (int e = 0; e < C::CPL; ++e) x[e] = v_ok ? __half2float(hv[e]) : 0.f;
      } else {
        const long long hi = vr * ngr + gv;
        const float s = KVQ_IN(c, KVQ_ARRAY_V_SCALE, p.scale[1] + hi, 2) ? __half2float(p.scale[1][hi]) : 0.f;
        const float z = nf4 ? 0.f
                      : (sym ? zsym
                             : (KVQ_IN(c, KVQ_ARRAY_V_ZERO, p.zero[1] + hi, 2) ? __half2float(p.zero[1][hi])
                                                                               : 0.f));
#pragma unroll
        for (int e = 0; e < C::CPL; ++e) {
          const int d = d0 + e;
          const uint32_t byte = v_ok ? rp[(d * BITS) >> 3] : 0u;
          const uint32_t q = (byte >> ((d * BITS) & 7)) & ((1u << BITS) - 1u);
          x[e] = nf4 ? lv_s[q] * s : ((float)q - z) * s;
        }
      }
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float pv = pw[t * GP + h];
#pragma unroll
        for (int e = 0; e < C::CPL; ++e) o[h][e] = fmaf(pv, x[e], o[h][e]);
      }
    }
    __syncwarp();  // before the next tile overwrites the probabilities
  }

  // ---- finish this warp, merge the warps ----
  if (bt_bad && p.status) atomicOr(p.status, KVQ_FLAG_BLOCK_TABLE);
#pragma unroll
  for (int h = 0; h < GP; ++h) {
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) l_lane[h] += __shfl_xor_sync(0xffffffffu, l_lane[h], o2);
#pragma unroll
    for (int e = 0; e < C::CPL; ++e) red[(warp * GP + h) * D + lane * C::CPL + e] = o[h][e];
    if (lane == 0) {
      ml[(warp * GP + h) * 2] = m_run[h];
      ml[(warp * GP + h) * 2 + 1] = l_lane[h];
    }
  }
  __syncthreads();

  const long long hq0 = (long long)b * p.Hq + (long long)kvh * G;
  for (int i = threadIdx.x; i < G * D; i += kWarps * 32) {
    const int h = i / D, d = i - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) M = fmaxf(M, ml[(w2 * GP + h) * 2]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) {
        const float f = exp2f(ml[(w2 * GP + h) * 2] - M);
        num = fmaf(f, red[(w2 * GP + h) * D + d], num);
        den = fmaf(f, ml[(w2 * GP + h) * 2 + 1], den);
      }
    }
    if (p.splits == 1) {
      if (KVQ_IN(c, KVQ_ARRAY_OUT, p.out + hq0 * D + i, 2))
        p.out[hq0 * D + i] = __float2half_rn(den > 0.f ? num / den : 0.f);
    } else {
      float* w = p.ws_o + ((hq0 + h) * p.splits + split) * D + d;
      if (KVQ_IN(c, KVQ_ARRAY_WORKSPACE, w, 4)) *w = num;
      if (d == 0) {
        float* mlo = p.ws_ml + ((hq0 + h) * p.splits + split) * 2;
        if (KVQ_IN(c, KVQ_ARRAY_WORKSPACE, mlo, 8)) {
          mlo[0] = M;
          mlo[1] = den;
        }
      }
    }
  }
}

template <int BITS, int D, int GP>
cudaError_t launch_cc_inst(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm) {
  const size_t smem = cc_smem_bytes<BITS, D, GP>();
  static KernelSetup setup;  // the shared-memory attribute and occupancy, once per device
  const cudaError_t e = setup_kernel(decode_cc_kernel<BITS, D, GP>, setup, kWarps * 32, smem,
                                     ctas_per_sm);
  if (e != cudaSuccess || ctas_per_sm) return e;
  const dim3 grid(p.splits, p.geom.Hkv, p.batch);
  // a plain launch: with programmatic serialization this kernel ran 2-7 %
  // slower (fp16, NF4 and INT2 caches on the 7B-class step)
  decode_cc_kernel<BITS, D, GP><<<grid, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

// head_dim and padded heads per KV head from the parameters
template <int BITS>
cudaError_t launch_cc_bits(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm) {
  int gp = 1;
  while (gp < p.G) gp <<= 1;
  const int D = p.geom.D;
#define KVQ_CC_GP(DD)                                                        \
  switch (gp) {                                                              \
    case 1: return launch_cc_inst<BITS, DD, 1>(p, stream, ctas_per_sm);      \
    case 2: return launch_cc_inst<BITS, DD, 2>(p, stream, ctas_per_sm);      \
    case 4: return launch_cc_inst<BITS, DD, 4>(p, stream, ctas_per_sm);      \
    case 8: return launch_cc_inst<BITS, DD, 8>(p, stream, ctas_per_sm);      \
    default: return launch_cc_inst<BITS, DD, 16>(p, stream, ctas_per_sm);    \
  }
  if (D == 64) { KVQ_CC_GP(64) }
  if (D == 128) { KVQ_CC_GP(128) }
  KVQ_CC_GP(256)
#undef KVQ_CC_GP
}

}  // namespace cc
}  // namespace kvq
