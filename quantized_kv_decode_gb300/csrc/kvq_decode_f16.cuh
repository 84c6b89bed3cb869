// Tensor-core split-K decode attention over fp16 caches, the unquantized
// comparator format (head_dim 64 / 128, up to 8 query heads per KV head).
//
// It computes the decode step of "Quantization & inference optimisation"
// ("Prefill, then decode": scores = K q / sqrt(d), softmax over every cached
// row, weighted V) on the fp16 rows themselves: no codes, scales or
// zero-points, so the work per byte is small and the kernel streams.
//
// One CTA per (split, KV head, sequence), 4 warps, each streaming its own
// 16-token tiles through a cp.async ring (K and V rows, 16-byte chunks
// XOR-swizzled by row so that every ldmatrix is conflict-free):
//  * scores: mma.m16n8k16 with A = q (rows = the KV head's query heads,
//    rows 8..15 empty) and B = K^T straight from the ring (ldmatrix of the
//    token rows); per 16 tokens two n-tiles of 8 tokens, head_dim / 16
//    k-blocks each;
//  * the accumulator layout (row = head, columns = tokens 2j, 2j + 1 of the
//    lane) is the B-operand layout of the weighted-V mma, so the
//    probabilities stay in the lanes that computed the scores;
//  * online softmax per head in log2 units with a lazily moved reference
//    maximum (rescale only when a tile exceeds it by 2^4);
//  * weighted V: A = V^T from the ring by ldmatrix.trans (rows = channels,
//    columns = tokens), B = the probabilities;
//  * the warps' (m, l, o) are merged in shared memory; the CTA writes the
//    output row (one split) or its partial for the merge kernel.
#pragma once

#include "kvq_decode_fast.cuh"

namespace kvq {
namespace f16 {

using fast::cp_async16;
using fast::cp_async_commit;
using fast::cp_async_wait;
using fast::ex2;
using fast::kSlack;
using fast::ldsm_x4;
using fast::ldsm_x4_t;
using fast::mma16816;
using fast::pack_h2;
using fast::pack_halves;
using fast::smem_u32;

constexpr int kWarps = 4;
constexpr int kTT = 16;  // tokens per warp tile

template <int D, int GP>
struct Cfg {
  static constexpr int ROWB = 2 * D;              // bytes per fp16 row
  static constexpr int CHUNKS = ROWB / 16;        // 16-byte chunks per row
  static constexpr int TILE = kTT * ROWB;         // K (or V) bytes of a tile
  static constexpr int STAGE = 2 * TILE;          // K then V
  static constexpr int KB = D / 16;               // score k-blocks
  static constexpr int MT = D / 16;               // V m-tiles
  // two CTAs per SM: about 96 KB of ring per CTA
  static constexpr int STAGES = (96 * 1024) / (kWarps * STAGE) > 6 ? 6 : (96 * 1024) / (kWarps * STAGE);
  static constexpr int WARP_BYTES = STAGES * STAGE;
  static_assert(STAGES >= 2, "at least two stages");
  static_assert(CHUNKS >= 8, "the swizzle needs 8 chunks per row");
  static_assert(GP <= 8, "heads fill rows 0..7 of the score mma");
  // byte offset of 16-byte chunk c of token row t in a K or V tile
  __device__ static __forceinline__ uint32_t at(int t, int c) {
    return (uint32_t)(t * ROWB + ((c ^ (t & 7)) << 4));
  }
};

template <int D, int GP>
__host__ __device__ constexpr size_t smem_bytes() {
  using C = Cfg<D, GP>;
  const size_t q = ((size_t)GP * D * 2 + 127) / 128 * 128;
  const size_t pipe = (size_t)kWarps * C::WARP_BYTES;
  const size_t merge = (size_t)kWarps * GP * (D + 2) * sizeof(float);
  const size_t masks = ((size_t)kWarps * C::STAGES * 4 + 15) / 16 * 16;
  return q + (pipe > merge ? pipe : merge) + masks;
}

template <int D, int GP>
__global__ void __launch_bounds__(kWarps * 32, 2) decode_f16_kernel(const DecodeParams p) {
  using C = Cfg<D, GP>;
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheGeom& geo = p.geom;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rho = lane >> 2, j = lane & 3;

  pdl_launch_dependents();
  pdl_wait();

  int L = seq_len_of(p, b);
  if (L < 0 || L > p.len_limit) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0 && p.status) atomicOr(p.status, KVQ_FLAG_SEQ_LEN);
    L = 0;
  }
  const int t0 = split * p.chunk;
  const int t1 = min(L, t0 + p.chunk);
  if (p.splits > 1 && t0 >= L) return;  // the merge reads splits < ceil(L / chunk) only

  // shared memory: [q fp16 GP x D][per warp: the ring][tile masks]; the CTA
  // merge reuses the ring region
  __half* q_s = reinterpret_cast<__half*>(smem);
  uint8_t* pipe = smem + ((GP * D * 2 + 127) / 128) * 128;
  const size_t region = (size_t)kWarps * C::WARP_BYTES > (size_t)kWarps * GP * (D + 2) * 4
                            ? (size_t)kWarps * C::WARP_BYTES
                            : (size_t)kWarps * GP * (D + 2) * 4;
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(pipe + region);
  const __half* qg = p.q + ((long long)b * p.Hq + (long long)kvh * G) * D;
  for (int i = threadIdx.x; i < GP * D; i += blockDim.x)
    q_s[i] = (i < G * D && KVQ_IN(geo, KVQ_ARRAY_Q, qg + i, 2)) ? qg[i] : __float2half_rn(0.f);
  __syncthreads();

  // A fragments: row rho = head rho (zero beyond G), k-slots 2j, 2j+1 and
  // 2j+8, 2j+9 of each k-block; rows 8..15 stay empty
  uint32_t qa[C::KB][2];
#pragma unroll
  for (int kb = 0; kb < C::KB; ++kb) {
    const __half* qh = q_s + (rho < GP ? rho : 0) * D + 16 * kb + 2 * j;
    qa[kb][0] = rho < GP ? pack_halves(qh[0], qh[1]) : 0u;
    qa[kb][1] = rho < GP ? pack_halves(qh[8], qh[9]) : 0u;
  }

  const uint8_t* kc_g = reinterpret_cast<const uint8_t*>(p.codes[0]);
  const uint8_t* vc_g = reinterpret_cast<const uint8_t*>(p.codes[1]);
  const int ntiles = t1 > t0 ? (t1 - t0 + kTT - 1) / kTT : 0;
  const int nmine = ntiles > warp ? (ntiles - warp + kWarps - 1) / kWarps : 0;
  const uint32_t ring = smem_u32(pipe + warp * C::WARP_BYTES);
  bool bt_bad = false;

  // issues this warp's tile `it` into its stage (an empty group past the end)
  auto issue = [&](int it) {
    if (it < nmine) {
      const int stage = it % C::STAGES;
      const int start = t0 + (warp + it * kWarps) * kTT;
      const int n = min(kTT, t1 - start);
      long long row = -1;
      if (lane < n) {
        row = token_row(geo, b, kvh, start + lane);
        bt_bad |= row < 0;
      }
      const uint32_t kd = ring + stage * C::STAGE, vd = kd + C::TILE;
#pragma unroll
      for (int k = 0; k < kTT * C::CHUNKS / 32; ++k) {
        const int c = lane + 32 * k;
        const int tok = c / C::CHUNKS, part = c % C::CHUNKS;
        const long long r = __shfl_sync(0xffffffffu, row, tok);
        const bool ok = r >= 0;
        const long long off = ok ? r * C::ROWB + part * 16 : 0;
        cp_async16(kd + C::at(tok, part), kc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_K_CODES, kc_g + off, 16));
        cp_async16(vd + C::at(tok, part), vc_g + off, ok && KVQ_IN(geo, KVQ_ARRAY_V_CODES, vc_g + off, 16));
      }
      const unsigned bad = __ballot_sync(0xffffffffu, lane >= kTT || row < 0);
      if (lane == 0) mask_s[warp * C::STAGES + stage] = bad;
    }
    cp_async_commit();
  };

  float o[C::MT][4];
#pragma unroll
  for (int m = 0; m < C::MT; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
  float m_ref = -INFINITY, l_run = 0.f;

#pragma unroll
  for (int s2 = 0; s2 < C::STAGES - 1; ++s2) issue(s2);

  for (int it = 0; it < nmine; ++it) {
    issue(it + C::STAGES - 1);
    cp_async_wait<C::STAGES - 1>();  // tile it
    __syncwarp();
    const int stage = it % C::STAGES;
    const uint32_t ks = ring + stage * C::STAGE, vs = ks + C::TILE;
    const unsigned bad = mask_s[warp * C::STAGES + stage];

    // ---- scores: n-tile nt = tokens 8 nt .. 8 nt + 7 ----
    float acc[2][2][4];  // [n-tile][chain: even / odd k-blocks]
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int u = 0; u < 2; ++u) acc[nt][u][0] = acc[nt][u][1] = acc[nt][u][2] = acc[nt][u][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c4 = 0; c4 < C::CHUNKS; c4 += 4) {
        // matrices: chunks c4 .. c4 + 3 (channels 8 c4 ..) of the n-tile's 8 rows
        uint32_t r0, r1, r2, r3;
        ldsm_x4(ks + C::at(8 * nt + (lane & 7), c4 + (lane >> 3)), r0, r1, r2, r3);
        const int kb = c4 / 2;  // chunks c4, c4+1: k-block kb; c4+2, c4+3: kb + 1
        mma16816(acc[nt][0], qa[kb][0], 0u, qa[kb][1], 0u, r0, r1);
        mma16816(acc[nt][1], qa[kb + 1][0], 0u, qa[kb + 1][1], 0u, r2, r3);
      }
    }
    // row rho (head rho), columns 2j, 2j+1 of each n-tile: tokens 8 nt + 2j + e
    float s[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 8 * nt + 2 * j + e;
        s[nt][e] = ((bad >> t) & 1u) ? -INFINITY : (acc[nt][0][e] + acc[nt][1][e]) * p.scale_log2;
      }

    // ---- online softmax per head (the 4 lanes of row rho) ----
    float mt = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const bool need = mt > m_ref + kSlack;
    const float m_next = need ? mt : m_ref;
    if (__any_sync(0xffffffffu, need)) {
      const float alpha = need ? ex2(m_ref - m_next) : 1.f;  // 0 on the first live tile
      l_run *= alpha;
      // o columns 2j, 2j+1 belong to heads 2j, 2j+1
      const float a0 = __shfl_sync(0xffffffffu, alpha, (2 * j) << 2);
      const float a1 = __shfl_sync(0xffffffffu, alpha, (2 * j + 1) << 2);
#pragma unroll
      for (int m = 0; m < C::MT; ++m) {
        o[m][0] *= a0; o[m][1] *= a1; o[m][2] *= a0; o[m][3] *= a1;
      }
    }
    m_ref = m_next;
    const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
    float pr[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = ex2(s[nt][0] - m_use);
      pr[nt][1] = ex2(s[nt][1] - m_use);
      l_run += pr[nt][0] + pr[nt][1];
    }
    // B of the weighted-V mma: k = tokens 2j, 2j+1 (n-tile 0) and 8 + 2j,
    // 9 + 2j (n-tile 1), n = head rho: the lane's own probabilities
    const uint32_t b0 = pack_h2(pr[0][0], pr[0][1]);
    const uint32_t b1 = pack_h2(pr[1][0], pr[1][1]);

    // ---- weighted V: m-tile m = channels 16 m .. 16 m + 15 ----
#pragma unroll
    for (int m = 0; m < C::MT; ++m) {
      // matrices: (channels 16m.., tokens 0-7), (16m+8.., 0-7), (16m.., 8-15), (16m+8.., 8-15)
      const int mi = lane >> 3;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vs + C::at(((mi >> 1) << 3) + (lane & 7), 2 * m + (mi & 1)), a0, a1, a2, a3);
      mma16816(o[m], a0, a1, a2, a3, b0, b1);
    }
    __syncwarp();  // the stage is refilled by the next issue
  }
  cp_async_wait<0>();

  // ---- this warp's partials, then the CTA merge ----
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  if (bt_bad && p.status) atomicOr(p.status, KVQ_FLAG_BLOCK_TABLE);
  __syncthreads();  // every warp is done with its ring
  float* red = reinterpret_cast<float*>(pipe);  // [warps][GP][D]
  float* ml = red + kWarps * GP * D;            // [warps][GP][2]
#pragma unroll
  for (int m = 0; m < C::MT; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int h = 2 * j + (e & 1);
      const int d = 16 * m + rho + ((e >> 1) << 3);
      if (h < GP) red[(warp * GP + h) * D + d] = o[m][e];
    }
  if (j == 0 && rho < GP) {
    ml[(warp * GP + rho) * 2] = m_ref;
    ml[(warp * GP + rho) * 2 + 1] = l_run;
  }
  __syncthreads();

  const long long hq0 = (long long)b * p.Hq + (long long)kvh * G;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
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
      if (KVQ_IN(geo, KVQ_ARRAY_OUT, p.out + hq0 * D + i, 2))
        p.out[hq0 * D + i] = __float2half_rn(den > 0.f ? num / den : 0.f);
    } else {
      float* w = p.ws_o + ((hq0 + h) * p.splits + split) * D + d;
      if (KVQ_IN(geo, KVQ_ARRAY_WORKSPACE, w, 4)) *w = num;
      if (d == 0) {
        float* mlo = p.ws_ml + ((hq0 + h) * p.splits + split) * 2;
        if (KVQ_IN(geo, KVQ_ARRAY_WORKSPACE, mlo, 8)) {
          mlo[0] = M;
          mlo[1] = den;
        }
      }
    }
  }
}

// Launches the instantiation, or with ctas_per_sm != nullptr only reports
// how many of its CTAs fit on one SM.
template <int D, int GP>
cudaError_t launch_inst(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm) {
  const size_t smem = smem_bytes<D, GP>();
  static KernelSetup setup;  // the shared-memory attribute and occupancy, once per device
  const cudaError_t e = setup_kernel(decode_f16_kernel<D, GP>, setup, kWarps * 32, smem, ctas_per_sm);
  if (e != cudaSuccess || ctas_per_sm) return e;
  return launch_pdl(decode_f16_kernel<D, GP>, dim3(p.splits, p.geom.Hkv, p.batch), dim3(kWarps * 32),
                    smem, stream, p);
}

// fp16 caches at head_dim 64 / 128 with at most 8 query heads per KV head;
// *handled is false for the other shapes
inline cudaError_t launch(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm, bool* handled) {
  *handled = true;
  int gp = 1;
  while (gp < p.G) gp <<= 1;
  const int D = p.geom.D;
#define KVQ_F16_GP(DD)                                                  \
  switch (gp) {                                                         \
    case 1: return launch_inst<DD, 1>(p, stream, ctas_per_sm);          \
    case 2: return launch_inst<DD, 2>(p, stream, ctas_per_sm);          \
    case 4: return launch_inst<DD, 4>(p, stream, ctas_per_sm);          \
    case 8: return launch_inst<DD, 8>(p, stream, ctas_per_sm);          \
    default: break;                                                     \
  }
  if (D == 64) { KVQ_F16_GP(64) }
  if (D == 128) { KVQ_F16_GP(128) }
#undef KVQ_F16_GP
  *handled = false;
  return cudaSuccess;
}

}  // namespace f16
}  // namespace kvq
