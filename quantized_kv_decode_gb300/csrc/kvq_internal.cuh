// Internal declarations shared by the CUDA translation units of libkvq.
// Nothing here is part of the public ABI (include/kvq.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/kvq.h"

namespace kvq {

// Token tile of the generic decode kernel and the alignment of split chunks:
// every split except the last covers a multiple of this many tokens.
constexpr int kChunkAlign = 64;
constexpr int kMaxGroupHeads = 16;  // query heads per KV head handled per CTA

// Debug builds (KVQ_DEBUG): the byte extent [lo, hi) of each caller array a
// launch may touch, indexed by kvq_array, and the status word to flag.  The
// host fills it from the descriptor and the call's sizes; it travels in the
// cache geometry so that every kernel and helper that addresses a caller
// array can check the access first.
struct DbgExtents {
  unsigned long long lo[KVQ_ARRAY_COUNT];
  unsigned long long hi[KVQ_ARRAY_COUNT];
  uint32_t* status;
};

// The kernels name K / V pairs and the prefetch regions by offset.
static_assert(KVQ_ARRAY_V_CODES == KVQ_ARRAY_K_CODES + 1 && KVQ_ARRAY_K_SCALE == 2 &&
                  KVQ_ARRAY_K_ZERO == 3 && KVQ_ARRAY_V_SCALE == 4 && KVQ_ARRAY_V_ZERO == 5 &&
                  KVQ_ARRAY_V_WINDOW == KVQ_ARRAY_K_WINDOW + 1 &&
                  KVQ_ARRAY_V_NEW == KVQ_ARRAY_K_NEW + 1,
              "kvq_array order");

#ifdef KVQ_DEBUG
// True when the n bytes at ptr lie inside array a's extent; otherwise flags
// KVQ_FLAG_OOB and returns false, and the caller skips the access.
__device__ __forceinline__ bool dbg_in(const DbgExtents& x, int a, const void* ptr,
                                       unsigned long long n) {
  const unsigned long long u = (unsigned long long)reinterpret_cast<uintptr_t>(ptr);
  if (u >= x.lo[a] && u + n <= x.hi[a]) return true;
  if (x.status) atomicOr(x.status, KVQ_FLAG_OOB);
  return false;
}
// KVQ_IN(geometry, kvq_array, pointer, bytes): may the access go ahead?
#define KVQ_IN(geo, a, ptr, n) (::kvq::dbg_in((geo).dbg, (a), (ptr), (n)))
#else
// (release: no check; the array id and pointer are only named, so that
// variables kept for the check count as used)
#define KVQ_IN(geo, a, ptr, n) ((void)(a), (void)(ptr), true)
#endif

// Geometry of one cache (K and V share it).
struct CacheGeom {
  int32_t bits;        // 4, 8 or 16
  int32_t D;           // head_dim
  int32_t g;           // group size (channels per scale/zero)
  int32_t ngroups;     // D / g (0 when bits == 16)
  int32_t row_bytes;   // bytes of codes per token row
  int32_t Hkv;
  int32_t layout;      // KVQ_DENSE / KVQ_PAGED
  int32_t slots;       // dense: capacity; paged: page size
  int32_t num_pages;   // paged only
  int32_t max_blocks;  // paged only
  int32_t sym;         // 1: symmetric codes (offset 2^(bits-1)), no zero arrays
  int32_t kch;         // 1: axis-aware cache (K per channel, fp16 sinks + residual)
  int32_t sink;        // axis-aware: fp16 sink tokens
  int32_t nf4;         // 1: 4-bit codes index the normal-quantile levels, no zero arrays
  const int32_t* block_table;
#ifdef KVQ_DEBUG
  DbgExtents dbg;
#endif
};

// Axis-aware caches: the window slot of position p, or -1 when p is stored
// quantized (L = tokens cached).  Sinks [0, min(S, L)), residual window
// [r0, L) with r0 = S + floor((L - S) / g) g.
__device__ __forceinline__ int window_slot(const CacheGeom& c, int L, int p) {
  const int S = min(c.sink, L);
  if (p < S) return p;
  const int r0 = S + ((L - S) / c.g) * c.g;
  return p >= r0 ? c.sink + (p - c.sink) % c.g : -1;
}

// Axis-aware caches.  Dense: a sequence's rows are positions 0 .. slots-1
// (the sink and window positions unused) and its K block j has header row
// j.  Paged: only the quantized region is paged, indexed by u = pos - sink;
// a page holds `slots` rows (a multiple of g, so a block never straddles
// pages), page i of sequence b is block_table[b][i], and a page's K header
// rows are its slots / g blocks.
// Code / V-header row of position pos >= sink (-1: unmapped page).
__device__ __forceinline__ long long kch_row(const CacheGeom& c, int b, int kvh, int pos) {
  if (c.layout == KVQ_DENSE) return ((long long)b * c.Hkv + kvh) * c.slots + pos;
  const int u = pos - c.sink;
  if (u < 0) return -1;
  const int blk = u / c.slots;
  if (blk >= c.max_blocks) return -1;
  const int32_t* e = c.block_table + (long long)b * c.max_blocks + blk;
  const int page = KVQ_IN(c, KVQ_ARRAY_BLOCK_TABLE, e, 4) ? __ldg(e) : -1;
  if (page < 0 || page >= c.num_pages) return -1;
  return ((long long)page * c.Hkv + kvh) * c.slots + (u - blk * c.slots);
}

// K header row of block j >= 0 (times D: the block's per-channel scales and
// zeros); -1 for an unmapped page.
__device__ __forceinline__ long long kch_hdr(const CacheGeom& c, int b, int kvh, int j) {
  const int bpp = c.slots / c.g;  // blocks per sequence (dense) or per page
  if (c.layout == KVQ_DENSE) return ((long long)b * c.Hkv + kvh) * bpp + j;
  const int blk = j / bpp;
  if (blk >= c.max_blocks) return -1;
  const int32_t* e = c.block_table + (long long)b * c.max_blocks + blk;
  const int page = KVQ_IN(c, KVQ_ARRAY_BLOCK_TABLE, e, 4) ? __ldg(e) : -1;
  if (page < 0 || page >= c.num_pages) return -1;
  return ((long long)page * c.Hkv + kvh) * bpp + (j - blk * bpp);
}

// Positions an axis-aware cache can hold per sequence.
__device__ __forceinline__ long long kch_capacity(const CacheGeom& c) {
  return c.layout == KVQ_DENSE ? (long long)c.slots : c.sink + (long long)c.slots * c.max_blocks;
}

// Row index of token `pos` of sequence `b`, KV head `kvh`, into the
// [..][row_bytes] codes array and the [..][ngroups] header arrays;
// -1 when the block table maps the token to no valid page.
__device__ __forceinline__ long long token_row(const CacheGeom& c, int b, int kvh,
                                               int pos) {
  if (c.layout == KVQ_DENSE) {
    return ((long long)b * c.Hkv + kvh) * c.slots + pos;
  }
  const int blk = pos / c.slots;
  const int off = pos - blk * c.slots;
  const int32_t* e = c.block_table + (long long)b * c.max_blocks + blk;
  const int page = KVQ_IN(c, KVQ_ARRAY_BLOCK_TABLE, e, 4) ? __ldg(e) : -1;
  if (page < 0 || page >= c.num_pages) return -1;
  return ((long long)page * c.Hkv + kvh) * c.slots + off;
}

struct AppendParams {
  CacheGeom geom;
  uint8_t* codes[2];     // K, V
  __half* scale[2];
  __half* zero[2];
  const __half* src[2];  // k_new, v_new: [batch][num_new][Hkv][D]
  __half* window[2];     // axis-aware caches: fp16 sinks + residual, K and V
  float nf4_mid[16];     // NF4: midpoints between consecutive levels (15 used)
  const int32_t* seq_lens_before;
  uint32_t* status;
  int32_t batch;
  int32_t num_new;
};

struct DecodeParams {
  CacheGeom geom;
  const uint8_t* codes[2];  // K, V
  const __half* scale[2];
  const __half* zero[2];
  const __half* q;          // [batch][Hq][D]
  const int32_t* seq_lens;  // [batch]
  __half* out;              // [batch][Hq][D]
  float* ws_o;              // [batch][Hq][splits][D]     (splits > 1)
  float* ws_ml;             // [batch][Hq][splits][2]      (splits > 1)
  uint32_t* status;
  int32_t batch;
  int32_t Hq;
  int32_t G;                // Hq / Hkv
  int32_t splits;
  int32_t chunk;            // tokens per split (multiple of kChunkAlign)
  int32_t len_limit;        // largest valid seq_len
  float scale_log2;         // softmax scale * log2(e)
  // fused append + decode: lengths before the step and the new token's K/V
  // ([batch][Hkv][D]); the attended length is lens_before + 1 (seq_lens unused)
  const int32_t* lens_before;
  const __half* new_kv[2];
  const __half* window[2];  // axis-aware caches: fp16 sinks + residual, K and V
  float nf4_level[16];      // NF4: the 16 levels (fp16 values as fp32)
  // Tensor-core kernel: grid index z is a rank in the longest-first order of
  // the batch instead of the sequence index (set for grids of more than one
  // wave, so that the longest sequences start first)
  int32_t longest_first;
  // Paged per-token caches whose code arrays hold fewer than 2^31 bytes: the
  // tensor-core kernel forms token rows and byte offsets in 32 bits
  int32_t rows32;
  // Fused step on an axis-aware cache with one split: each CTA of the
  // tensor-core kernel first appends its (sequence, KV head)'s new token
  // (window slot, or the block it completes), then attends
  int32_t kch_append;
  // Split calls of the tensor-core kernel: every split CTA writes its
  // partial, a split past the sequence's end the marker m = -inf, so the
  // merge reads all splits without the lengths
  int32_t merge_all;
};

// lens[b] (a length array of the call), or `bad` when a debug build finds the
// read outside the array.
__device__ __forceinline__ int checked_len(const CacheGeom& c, const int32_t* lens, int b, int bad) {
  return KVQ_IN(c, KVQ_ARRAY_SEQ_LENS, lens + b, 4) ? __ldg(lens + b) : bad;
}

// Tokens to attend over for sequence b (-1 for a length that cannot be formed).
__device__ __forceinline__ int seq_len_of(const DecodeParams& p, int b) {
  if (p.lens_before) {
    const int x = checked_len(p.geom, p.lens_before, b, -1);
    return (x < 0 || x == 0x7fffffff) ? -1 : x + 1;
  }
  return checked_len(p.geom, p.seq_lens, b, -1);
}

// The sequence of rank r in a longest-first order of the batch: sequences
// are put in 128 buckets of attended length (an unusable length counts as 0),
// the buckets taken longest first and a bucket's sequences by index, so the
// ranks are a permutation.  O(batch) per CTA: a histogram, a scan of the
// buckets by one warp, and a ballot search for the r-th sequence of its
// bucket.  Every thread of the CTA calls it; `scratch` is shared memory for
// 132 ints and batch bytes, free again on return.
constexpr int kLongestFirstMaxBatch = 4096;
constexpr int kOrderBuckets = 128;
__device__ __forceinline__ int longest_first_seq(const DecodeParams& p, int r, int* scratch) {
  const int B = p.batch;
  int* hist = scratch;               // [kOrderBuckets]
  int* res = scratch + kOrderBuckets;  // bucket of rank r, rank within it, sequence
  uint8_t* bkt = reinterpret_cast<uint8_t*>(scratch + kOrderBuckets + 4);  // [B]
  for (int i = threadIdx.x; i < kOrderBuckets; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const long long span = (long long)max(p.len_limit, 0) + 1;
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    const int L = seq_len_of(p, i);
    const int Lc = (L < 0 || L > p.len_limit) ? 0 : L;
    const int k = (int)((long long)Lc * kOrderBuckets / span);
    bkt[i] = (uint8_t)k;
    atomicAdd(hist + k, 1);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    // lane l holds buckets 127 - 4l ... 124 - 4l (longest first)
    int cnt[4], sum = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      cnt[e] = hist[kOrderBuckets - 1 - (4 * lane + e)];
      sum += cnt[e];
    }
    int inc = sum;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o2);
      if (lane >= o2) inc += y;
    }
    int before = inc - sum;  // sequences in longer buckets
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (r >= before && r < before + cnt[e]) {
        res[0] = kOrderBuckets - 1 - (4 * lane + e);
        res[1] = r - before;
      }
      before += cnt[e];
    }
    __syncwarp();
    const int kz = res[0];
    int k = res[1];
    for (int base = 0; base < B; base += 32) {  // the k-th sequence of bucket kz
      const int i = base + lane;
      const unsigned m = __ballot_sync(0xffffffffu, i < B && bkt[i] == kz);
      const int n = __popc(m);
      if (k < n) {  // warp-uniform
        unsigned mm = m;
        for (int t = 0; t < k; ++t) mm &= mm - 1;
        if (lane == 0) res[2] = base + __ffs(mm) - 1;
        break;
      }
      k -= n;
    }
  }
  __syncthreads();
  const int b = res[2];
  __syncthreads();
  return b;
}

// Programmatic dependent launch.  The library's kernels (all but the
// CUDA-core decode kernel) are launched with programmatic stream
// serialization: the next kernel of the stream may
// start launching once all CTAs have passed pdl_launch_dependents, and each
// kernel reads or writes caller memory only after pdl_wait, which returns
// when the previous kernel has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

template <typename Params>
cudaError_t launch_pdl(void (*kernel)(Params), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Devices whose one-time kernel set-up the library caches.
constexpr int kMaxDevices = 64;

// Identifier of the current thread's CUDA context (the driver never reuses
// one), or 0 when none is current or it cannot be read.  Set-up that lives in
// a context (kernel attributes, the address of a module symbol) is cached
// together with this identifier and redone when it changes, e.g. after
// cudaDeviceReset.
unsigned long long current_context_id();

// One-time set-up of a kernel whose dynamic shared memory has a fixed size:
// the attribute that allows that size and the CTAs per SM it leaves, cached
// per device (a function-local static per kernel instantiation).
struct KernelSetup {
  std::atomic<unsigned long long> ctx[kMaxDevices];
  std::atomic<int> occ[kMaxDevices];
};

// Raises the kernel's dynamic shared-memory limit to `smem` and reports its
// resident CTAs per SM for `threads` threads, once per device and context;
// later calls read the cache.
template <typename Kernel>
cudaError_t setup_kernel(Kernel kernel, KernelSetup& s, int threads, size_t smem,
                         int* ctas_per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  const bool cached = ctx != 0 && dev >= 0 && dev < kMaxDevices;
  if (cached && s.ctx[dev].load(std::memory_order_acquire) == ctx) {
    if (ctas_per_sm) *ctas_per_sm = s.occ[dev].load(std::memory_order_relaxed);
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (cached) {
    s.occ[dev].store(n, std::memory_order_relaxed);
    s.ctx[dev].store(ctx, std::memory_order_release);
  }
  if (ctas_per_sm) *ctas_per_sm = n;
  return cudaSuccess;
}

// Launchers (return a CUDA error code; the caller maps it to kvq_status).
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_append_kivi(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_decode_generic(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_cc_b2(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm);
cudaError_t launch_decode_cc_b4(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm);
cudaError_t launch_decode_cc_b8(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm);
cudaError_t launch_decode_cc_b16(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm);
// Tensor-core kernel for INT4/INT8 caches; *handled is false when the shape
// (head_dim, groups, padded heads per KV head `gp`) has no instantiation.
// With occ != nullptr nothing is launched: *occ receives the CTAs per SM.
cudaError_t launch_decode_fast_int4(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                                    int* occ);
cudaError_t launch_decode_fast_int4_sym(const DecodeParams& p, int gp, cudaStream_t s,
                                        bool* handled, int* occ);
// INT2 caches, head_dim 128
cudaError_t launch_decode_fast_int2(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                                    int* occ);
// NF4 caches (with a symmetric level table: the caller checks it)
cudaError_t launch_decode_fast_nf4(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                                   int* occ);
cudaError_t launch_decode_fast_int8_sym(const DecodeParams& p, int gp, cudaStream_t s,
                                        bool* handled, int* occ);
cudaError_t launch_decode_fast_int4_kch(const DecodeParams& p, int gp, cudaStream_t s,
                                        bool* handled, int* occ);
// (paged axis-aware caches)
cudaError_t launch_decode_fast_int4_kch_paged(const DecodeParams& p, int gp, cudaStream_t s,
                                              bool* handled, int* occ);
cudaError_t launch_decode_fast_int8_kch(const DecodeParams& p, int gp, cudaStream_t s,
                                        bool* handled, int* occ);
// (paged axis-aware caches)
cudaError_t launch_decode_fast_int8_kch_paged(const DecodeParams& p, int gp, cudaStream_t s,
                                              bool* handled, int* occ);
cudaError_t launch_decode_fast_int8(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                                    int* occ);
int generic_ctas_per_sm(const DecodeParams& p);

// Size of the workspace for `splits` splits (0 when splits == 1).
size_t workspace_bytes(int64_t batch, int64_t Hq, int64_t D, int64_t splits);
void workspace_carve(void* ws, int64_t batch, int64_t Hq, int64_t D, int64_t splits,
                     float** ws_o, float** ws_ml);

}  // namespace kvq
