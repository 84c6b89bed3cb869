// Append into axis-aware caches: K grouped per channel over blocks of g
// tokens, V per token, fp16 sinks and residual window.
//
// "What actually happens when you quantize a KV cache", section 3 step 7
// ("axis choice": a K group is one channel across consecutive tokens, so a
// hot channel shares its scale with no other; V keeps per-token groups;
// per-channel K needs a few tokens buffered until a group fills, kept in an
// fp16 residual window; "sinks": the first tokens stay fp16) and section 7.
// The quantizer itself is the asymmetric one of section 3 steps 2-5 and
// section 4 (group_params / group_encode / quantize8 in kvq_quant.cuh), so a
// K group here is exactly a per-token group with its axis turned.
//
// An append of several tokens is two launches in stream order:
//  1. kivi_block_kernel: every block that this append completes is
//     quantized, reading the tokens already in the residual window and the
//     new ones;
//  2. kivi_window_kernel: sink tokens and the tokens left in the (new)
//     residual window are written to their fp16 slots.  It runs second
//     because its slots may be the ones launch 1 reads.
// A one-token append (the decode step) is one launch, kivi_step_kernel.
#include "kvq_kivi.cuh"

namespace kvq {
namespace {

constexpr int kBlockThreads = 128;

__device__ __forceinline__ KiviIO kivi_io(const AppendParams& p) {
  KiviIO io;
  io.geom = &p.geom;
  for (int w = 0; w < 2; ++w) {
    io.codes[w] = p.codes[w];
    io.scale[w] = p.scale[w];
    io.zero[w] = p.zero[w];
    io.src[w] = p.src[w];
    io.window[w] = p.window[w];
  }
  io.status = p.status;
  io.num_new = p.num_new;
  return io;
}

template <int BITS>
__global__ void __launch_bounds__(kBlockThreads) kivi_block_kernel(const AppendParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const CacheGeom& c = p.geom;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int S = c.sink, g = c.g;
  const int p0 = checked_len(p.geom, p.seq_lens_before, b, -1);
  const int n = p.num_new;
  if (p0 < 0) return;  // flagged by the window kernel
  // the block holding the first new token (or block 0), then the next ones
  const int j = (p0 <= S ? 0 : (p0 - S) / g) + blockIdx.x;
  const long long start = (long long)S + (long long)j * g;
  const long long end = start + g - 1;               // last position of the block
  if (end < p0 || end > (long long)p0 + n - 1) return;  // not completed by this append
  if (end >= kch_capacity(c)) {
    if (threadIdx.x == 0 && p.status) atomicOr(p.status, KVQ_FLAG_SEQ_LEN);
    return;
  }
  kivi_quantize_block<BITS>(kivi_io(p), b, kvh, j, start, p0);
}

// One-token append in one launch, one CTA per (KV head, sequence): the token
// either completes its block (quantized here, window rows read) or goes to
// its fp16 slot (a sink or the residual ring).  The two never meet within a
// sequence, so no second launch is needed to order them.
template <int BITS>
__global__ void __launch_bounds__(kBlockThreads) kivi_step_kernel(const AppendParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int kvh = blockIdx.y, b = blockIdx.z;
  kivi_append_one<BITS>(kivi_io(p), b, kvh, checked_len(p.geom, p.seq_lens_before, b, -1));
}

// Sinks and the residual window left after this append: one thread per
// 16-byte chunk of a new token's K and V.
__global__ void __launch_bounds__(256) kivi_window_kernel(const AppendParams p) {
  pdl_launch_dependents();
  pdl_wait();  // the block kernel reads the slots written here
  const CacheGeom& c = p.geom;
  const int chunks = c.D / 8;
  const long long units = (long long)p.batch * p.num_new * c.Hkv * chunks;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int ch = (int)(u % chunks);
  long long r = u / chunks;
  const int kvh = (int)(r % c.Hkv);
  r /= c.Hkv;
  const int t = (int)(r % p.num_new);
  const int b = (int)(r / p.num_new);
  const int p0 = checked_len(p.geom, p.seq_lens_before, b, -1);
  const long long q = (long long)p0 + t;
  if (p0 < 0 || q >= kch_capacity(c)) {
    if (ch == 0 && kvh == 0 && p.status) atomicOr(p.status, KVQ_FLAG_SEQ_LEN);
    return;
  }
  // the cache holds min(p0 + num_new, capacity) tokens after this append
  const int slot = window_slot(c, (int)min((long long)p0 + p.num_new, kch_capacity(c)), (int)q);
  if (slot < 0) return;  // quantized by the block kernel
  const long long bh = (long long)b * c.Hkv + kvh;
  const long long src = (((long long)b * p.num_new + t) * c.Hkv + kvh) * c.D + ch * 8;
  const long long dst = (bh * (c.sink + c.g) + slot) * c.D + ch * 8;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const __half* from = p.src[which] + src;
    __half* to = p.window[which] + dst;
    if (KVQ_IN(c, which ? KVQ_ARRAY_V_NEW : KVQ_ARRAY_K_NEW, from, 16) &&
        KVQ_IN(c, which ? KVQ_ARRAY_V_WINDOW : KVQ_ARRAY_K_WINDOW, to, 16))
      *reinterpret_cast<uint4*>(to) = *reinterpret_cast<const uint4*>(from);
  }
}

}  // namespace

cudaError_t launch_append_kivi(const AppendParams& p, cudaStream_t stream) {
  const CacheGeom& c = p.geom;
  if (p.batch == 0 || p.num_new == 0) return cudaSuccess;
  // blocks one append can complete: the one holding its first token and
  // every later one it reaches
  if (p.num_new == 1) {
    const dim3 grid(1, c.Hkv, p.batch);
    return c.bits == 4 ? launch_pdl(kivi_step_kernel<4>, grid, dim3(kBlockThreads), 0, stream, p)
                       : launch_pdl(kivi_step_kernel<8>, grid, dim3(kBlockThreads), 0, stream, p);
  }
  const long long nblk = (long long)(p.num_new + c.g - 1) / c.g + 1;
  const dim3 grid1((unsigned)nblk, c.Hkv, p.batch);
  cudaError_t e = c.bits == 4 ? launch_pdl(kivi_block_kernel<4>, grid1, dim3(kBlockThreads), 0, stream, p)
                              : launch_pdl(kivi_block_kernel<8>, grid1, dim3(kBlockThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  const long long units = (long long)p.batch * p.num_new * c.Hkv * (c.D / 8);
  return launch_pdl(kivi_window_kernel, dim3((unsigned)((units + 255) / 256)), dim3(256), 0, stream, p);
}

}  // namespace kvq
