// Generic split-K decode attention (CUDA cores) and the log-sum-exp merge.
//
// The generic kernel covers every shape the ABI accepts (INT4/INT8/fp16
// caches, any group size, head_dim 64/128/256, up to 16 query heads per KV
// head, dense or paged).  It keeps the plain structure of the decode step of
// "Quantization & inference optimisation" ("Prefill, then decode": scores =
// K q / sqrt(d), softmax, weighted V) in tiles of 64 tokens with an online
// softmax, dequantizing x_hat = (q - z) * s element by element in fp32
// ("What actually happens when you quantize a KV cache", section 3 step 3).
// The tensor-core kernel (kvq_decode_fast.cuh) is the fast path for the
// common shapes; both write the same partials, merged by merge_kernel.
//
// Work unit: one CTA per (split, KV head, sequence); the split covers
// tokens [split*chunk, min(len, (split+1)*chunk)).  Scores and softmax
// statistics are kept in the log2 domain (scores pre-multiplied by log2 e)
// so that exp2f serves both the kernel and the merge.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 128;
constexpr int kTile = 64;

// A caller array element, or 0 when a debug build finds it outside the array
template <typename T>
__device__ __forceinline__ T checked_at(const CacheGeom& c, int a, const T* ptr) {
  return KVQ_IN(c, a, ptr, sizeof(T)) ? *ptr : T(0);
}
__device__ __forceinline__ float checked_half(const CacheGeom& c, int a, const __half* ptr) {
  return KVQ_IN(c, a, ptr, 2) ? __half2float(*ptr) : 0.f;
}

// K (which = 0) or V (which = 1); nf4_level: the NF4 level table, or null
// for uniform codes
template <int BITS>
__device__ __forceinline__ float dequant(int which, const uint8_t* codes, const __half* scale,
                                         const __half* zero, const CacheGeom& c,
                                         long long row, int d, const float* nf4_level) {
  const int a_codes = which ? KVQ_ARRAY_V_CODES : KVQ_ARRAY_K_CODES;
  if constexpr (BITS == 16) {
    return checked_half(c, a_codes, reinterpret_cast<const __half*>(codes + row * c.row_bytes) + d);
  } else {
    const uint8_t* r = codes + row * c.row_bytes;
    int q;
    if constexpr (BITS == 2) {
      q = (checked_at(c, a_codes, r + (d >> 2)) >> (2 * (d & 3))) & 3;
    } else if constexpr (BITS == 4) {
      const uint8_t byte = checked_at(c, a_codes, r + (d >> 1));
      q = (d & 1) ? (byte >> 4) : (byte & 15);
    } else {
      q = checked_at(c, a_codes, r + d);
    }
    const long long h = row * c.ngroups + d / c.g;
    const float s = checked_half(c, which ? KVQ_ARRAY_V_SCALE : KVQ_ARRAY_K_SCALE, scale + h);
    if (nf4_level) return nf4_level[q] * s;
    const float z = c.sym ? (float)(1 << (BITS - 1))
                          : checked_half(c, which ? KVQ_ARRAY_V_ZERO : KVQ_ARRAY_K_ZERO, zero + h);
    return ((float)q - z) * s;
  }
}

// Channel d of K (which = 0) or V (which = 1) at position pos (cache row
// `row`) of a sequence of L tokens.  Axis-aware caches read sinks and the
// residual window as fp16 and K blocks with per-channel headers.
template <int BITS>
__device__ __forceinline__ float load_kv(const DecodeParams& p, int which, int b, int kvh, int L,
                                         int pos, long long row, int d) {
  const CacheGeom& c = p.geom;
  if constexpr (BITS != 16) {
    if (c.kch) {
      const long long bh = (long long)b * c.Hkv + kvh;
      const int slot = window_slot(c, L, pos);
      if (slot >= 0)
        return checked_half(c, which ? KVQ_ARRAY_V_WINDOW : KVQ_ARRAY_K_WINDOW,
                            p.window[which] + (bh * (c.sink + c.g) + slot) * c.D + d);
      if (which == 0) {
        const uint8_t* r = p.codes[0] + row * c.row_bytes;
        const uint8_t byte = checked_at(c, KVQ_ARRAY_K_CODES, r + (BITS == 4 ? d >> 1 : d));
        const float q = BITS == 4 ? (float)((d & 1) ? (byte >> 4) : (byte & 15)) : (float)byte;
        const long long h = kch_hdr(c, b, kvh, (pos - c.sink) / c.g) * c.D + d;
        return (q - checked_half(c, KVQ_ARRAY_K_ZERO, p.zero[0] + h)) *
               checked_half(c, KVQ_ARRAY_K_SCALE, p.scale[0] + h);
      }
    }
  }
  return dequant<BITS>(which, p.codes[which], p.scale[which], p.zero[which], c, row, d,
                       c.nf4 ? p.nf4_level : nullptr);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) decode_generic_kernel(const DecodeParams p) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float smem[];
  const CacheGeom& c = p.geom;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.G, D = c.D;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  float* q_s = smem;                  // [G][D]
  float* o_s = q_s + G * D;           // [G][D]
  float* p_s = o_s + G * D;           // [G][kTile] scores, then probabilities
  float* m_s = p_s + G * kTile;       // [G]
  float* l_s = m_s + G;               // [G]
  float* a_s = l_s + G;               // [G]
  long long* row_s = reinterpret_cast<long long*>(a_s + ((G + 1) & ~1));  // [kTile]

  int L = seq_len_of(p, b);
  const bool bad_len = (L < 0 || L > p.len_limit);
  if (bad_len) {
    if (tid == 0 && split == 0 && kvh == 0 && p.status) atomicOr(p.status, KVQ_FLAG_SEQ_LEN);
    L = 0;
  }
  const int t0 = split * p.chunk;
  const int t1 = min(L, t0 + p.chunk);
  if (p.splits > 1 && t0 >= L) return;  // the merge reads splits < ceil(L / chunk) only

  const __half* qg = p.q + ((long long)b * p.Hq + (long long)kvh * G) * D;
  for (int i = tid; i < G * D; i += kThreads) {
    q_s[i] = checked_half(c, KVQ_ARRAY_Q, qg + i);
    o_s[i] = 0.f;
  }
  if (tid < G) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  __syncthreads();

  for (int ts = t0; ts < t1; ts += kTile) {
    const int n = min(kTile, t1 - ts);

    // scores: one warp per token, lanes across channels
    for (int j = warp; j < n; j += kThreads / 32) {
      // axis-aware caches: window positions read the fp16 window (any row
      // >= 0 marks them live); the quantized ones map through kch_row
      const long long row = !c.kch ? token_row(c, b, kvh, ts + j)
                            : (window_slot(c, L, ts + j) >= 0 ? 0 : kch_row(c, b, kvh, ts + j));
      float part[kMaxGroupHeads];
#pragma unroll
      for (int h = 0; h < kMaxGroupHeads; ++h) part[h] = 0.f;
      if (row >= 0) {
        for (int d = lane; d < D; d += 32) {
          const float k = load_kv<BITS>(p, 0, b, kvh, L, ts + j, row, d);
#pragma unroll
          for (int h = 0; h < kMaxGroupHeads; ++h)
            if (h < G) part[h] = fmaf(q_s[h * D + d], k, part[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < kMaxGroupHeads; ++h) {
        if (h < G) {
          float v = part[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) p_s[h * kTile + j] = (row >= 0) ? v * p.scale_log2 : -INFINITY;
        }
      }
      if (lane == 0) {
        row_s[j] = row;
        if (row < 0 && p.status) atomicOr(p.status, KVQ_FLAG_BLOCK_TABLE);
      }
    }
    __syncthreads();

    // online softmax update, one thread per query head
    if (tid < G) {
      float* ps = p_s + tid * kTile;
      float mt = -INFINITY;
      for (int j = 0; j < n; ++j) mt = fmaxf(mt, ps[j]);
      const float m_old = m_s[tid];
      const float m_new = fmaxf(m_old, mt);
      float alpha = 1.f, lsum = 0.f;
      if (m_new == -INFINITY) {
        for (int j = 0; j < n; ++j) ps[j] = 0.f;
      } else {
        alpha = exp2f(m_old - m_new);
        for (int j = 0; j < n; ++j) {
          const float e = exp2f(ps[j] - m_new);
          ps[j] = e;
          lsum += e;
        }
      }
      m_s[tid] = m_new;
      l_s[tid] = l_s[tid] * alpha + lsum;
      a_s[tid] = alpha;
    }
    __syncthreads();

    // weighted V: each thread owns (head, channel) outputs
    for (int i = tid; i < G * D; i += kThreads) {
      const int h = i / D, d = i - h * D;
      float acc = o_s[i] * a_s[h];
      const float* ps = p_s + h * kTile;
      for (int j = 0; j < n; ++j) {
        const long long row = row_s[j];
        if (row < 0) continue;
        acc = fmaf(ps[j], load_kv<BITS>(p, 1, b, kvh, L, ts + j, row, d), acc);
      }
      o_s[i] = acc;
    }
    __syncthreads();
  }

  const long long hq0 = (long long)b * p.Hq + (long long)kvh * G;
  if (p.splits == 1) {
    for (int i = tid; i < G * D; i += kThreads) {
      const int h = i / D;
      const float l = l_s[h];
      if (KVQ_IN(c, KVQ_ARRAY_OUT, p.out + hq0 * D + i, 2))
        p.out[hq0 * D + i] = __float2half_rn(l > 0.f ? o_s[i] / l : 0.f);
    }
  } else {
    for (int i = tid; i < G * D; i += kThreads) {
      const int h = i / D, d = i - h * D;
      float* w = p.ws_o + ((hq0 + h) * p.splits + split) * D + d;
      if (KVQ_IN(c, KVQ_ARRAY_WORKSPACE, w, 4)) *w = o_s[i];
    }
    if (tid < G) {
      float* ml = p.ws_ml + ((hq0 + tid) * p.splits + split) * 2;
      if (KVQ_IN(c, KVQ_ARRAY_WORKSPACE, ml, 8)) {
        ml[0] = m_s[tid];
        ml[1] = l_s[tid];
      }
    }
  }
}

// out[b][h] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits
// that hold tokens of sequence b.  One CTA per (b, h), one thread per
// channel.  The splits go in batches of kMergeBatch whose loads are all
// issued before any is used, then one rescale per batch, so a call pays
// about one memory latency per batch (most calls: one batch).  After the
// tensor-core kernel (merge_all) every split carries a partial or the
// marker m = -inf, and the merge needs no length: a marked split's o is
// loaded but not used.  After the others only the ceil(len / chunk) splits
// that hold tokens are read.
constexpr int kMergeBatch = 16;
__global__ void __launch_bounds__(256) merge_kernel(const DecodeParams p) {
  pdl_launch_dependents();
  pdl_wait();  // the partials of the decode kernel before it
  const long long rowid = blockIdx.x;  // b * Hq + h
  const int b = (int)(rowid / p.Hq);
  const int D = p.geom.D;
  const int d = threadIdx.x;
  int nv = p.splits;
  if (!p.merge_all) {
    const int L = seq_len_of(p, b);
    nv = (L <= 0 || L > p.len_limit) ? 0 : (L + p.chunk - 1) / p.chunk;
  }
  const float* ml = p.ws_ml + rowid * p.splits * 2;
  const float* o = p.ws_o + rowid * p.splits * D + d;
  float M = -INFINITY, num = 0.f, den = 0.f;
  for (int s0 = 0; s0 < nv; s0 += kMergeBatch) {
    float m[kMergeBatch], l[kMergeBatch], x[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int s = s0 + u;
      m[u] = -INFINITY;
      l[u] = 0.f;
      x[u] = 0.f;
      if (s < nv && KVQ_IN(p.geom, KVQ_ARRAY_WORKSPACE, ml + 2 * s, 8) &&
          KVQ_IN(p.geom, KVQ_ARRAY_WORKSPACE, o + (long long)s * D, 4)) {
        const float2 v = *reinterpret_cast<const float2*>(ml + 2 * s);
        m[u] = v.x;
        l[u] = v.y;
        x[u] = o[(long long)s * D];  // loaded with m, l: one latency
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) Mn = fmaxf(Mn, m[u]);
    if (Mn == -INFINITY) continue;
    const float a = exp2f(M - Mn);  // 0 while nothing is merged yet
    num *= a;
    den *= a;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      // a split with no live token (or the marker) adds nothing; its o may
      // be a stale value of any bits, so it is not multiplied in
      if (m[u] == -INFINITY) continue;
      const float f = exp2f(m[u] - Mn);
      num = fmaf(f, x[u], num);
      den = fmaf(f, l[u], den);
    }
    M = Mn;
  }
  if (d < D && KVQ_IN(p.geom, KVQ_ARRAY_OUT, p.out + rowid * D + d, 2))
    p.out[rowid * D + d] = __float2half_rn(den > 0.f ? num / den : 0.f);
}

}  // namespace

namespace {
// the CUDA-core kernel of kvq_decode_cc.cuh for every cache except the
// axis-aware ones, which read per element through load_kv (kernel above)
cudaError_t launch_cc(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm) {
  switch (p.geom.bits) {
    case 2: return launch_decode_cc_b2(p, stream, ctas_per_sm);
    case 4: return launch_decode_cc_b4(p, stream, ctas_per_sm);
    case 8: return launch_decode_cc_b8(p, stream, ctas_per_sm);
    default: return launch_decode_cc_b16(p, stream, ctas_per_sm);
  }
}
}  // namespace

cudaError_t launch_decode_generic(const DecodeParams& p, cudaStream_t stream) {
  if (!p.geom.kch) return launch_cc(p, stream, nullptr);
  const int G = p.G, D = p.geom.D;
  const size_t smem = sizeof(float) * (2 * G * D + G * kTile + 3 * G + 1) +
                      sizeof(long long) * (kTile + 1);
  const dim3 grid(p.splits, p.geom.Hkv, p.batch);
  cudaError_t e = cudaSuccess;
  switch (p.geom.bits) {
    case 2:
      e = cudaFuncSetAttribute(decode_generic_kernel<2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) e = launch_pdl(decode_generic_kernel<2>, grid, dim3(kThreads), smem, stream, p);
      break;
    case 4:
      e = cudaFuncSetAttribute(decode_generic_kernel<4>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) e = launch_pdl(decode_generic_kernel<4>, grid, dim3(kThreads), smem, stream, p);
      break;
    case 8:
      e = cudaFuncSetAttribute(decode_generic_kernel<8>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) e = launch_pdl(decode_generic_kernel<8>, grid, dim3(kThreads), smem, stream, p);
      break;
    default:
      e = cudaFuncSetAttribute(decode_generic_kernel<16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) e = launch_pdl(decode_generic_kernel<16>, grid, dim3(kThreads), smem, stream, p);
      break;
  }
  return e;
}

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.batch * p.Hq;
  return launch_pdl(merge_kernel, dim3((unsigned)rows), dim3(p.geom.D), 0, stream, p);
}

int generic_ctas_per_sm(const DecodeParams& p) {
  if (!p.geom.kch) {
    int n = 0;
    return launch_cc(p, nullptr, &n) == cudaSuccess ? n : 0;
  }
  const int G = p.G, D = p.geom.D;
  const size_t smem = sizeof(float) * (2 * G * D + G * kTile + 3 * G + 1) +
                      sizeof(long long) * (kTile + 1);
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (p.geom.bits) {
    case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_generic_kernel<2>, kThreads, smem); break;
    case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_generic_kernel<4>, kThreads, smem); break;
    case 8: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_generic_kernel<8>, kThreads, smem); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_generic_kernel<16>, kThreads, smem); break;
  }
  return (e == cudaSuccess && n > 0) ? n : 1;
}

}  // namespace kvq
