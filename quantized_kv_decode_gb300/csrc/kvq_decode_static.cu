// kvq_decode_attn_static_ws: decode attention whose split scratch lives in a
// fixed buffer inside the library instead of a caller-provided workspace.
//
// Who needs it: a caller that must not allocate device memory around a
// decode call. Examples are a host whose device allocator cannot be reached
// from the code that issues the call (a plugin handed only its input and
// output buffers), or code that must keep its memory footprint fixed after
// start-up. Such a caller cannot honour kvq_decode_workspace_size() when the
// split planner asks for scratch. This entry point takes that scratch from
// a static device array of KVQ_STATIC_WORKSPACE_BYTES instead.
//
// The computation is kvq_decode_attn's: the same planner, kernels and merge,
// with the array below passed as the workspace.
#include <mutex>

#include <cuda_runtime.h>

#include "kvq_internal.cuh"

namespace {

// The split partials ([batch][heads][splits][head_dim] o, then m and l) of
// one call. Every (m, l) a merge reads is written earlier in the same call,
// and an o is used only when its split's m says it holds tokens, so nothing
// here has to start at zero and nothing is cleared.
__device__ __align__(256) unsigned char g_split_scratch[KVQ_STATIC_WORKSPACE_BYTES];

std::mutex g_setup_mutex;
struct ScratchAddress {
  unsigned long long ctx;  // the context the address belongs to
  void* ptr;
};
ScratchAddress g_scratch[kvq::kMaxDevices] = {};

// Device address of g_split_scratch on the current device. It is looked up
// with that device current on the first call made there, which loads this
// library's device code on that device if the CUDA runtime has not done so
// yet, and again whenever the device's context has changed since (after a
// cudaDeviceReset the module, and so the array, lives at a new address).
kvq_status scratch_on_current_device(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kvq::kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  const unsigned long long ctx = kvq::current_context_id();
  if (!g_scratch[dev].ptr || ctx == 0 || g_scratch[dev].ctx != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
    // (the lookup made the context current if it was not yet)
    g_scratch[dev].ctx = kvq::current_context_id();
    g_scratch[dev].ptr = p;
  }
  *ptr = g_scratch[dev].ptr;
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_static_ws(const kvq_cache_desc* desc,
                                                const kvq_cache* cache, int32_t batch,
                                                int32_t num_q_heads, const uint16_t* q,
                                                const int32_t* seq_lens, int32_t max_seq_len,
                                                int32_t num_splits, float softmax_scale,
                                                uint16_t* out, uint32_t* dev_status,
                                                void* stream) {
  void* scratch = nullptr;
  const kvq_status st = scratch_on_current_device(&scratch);
  if (st != KVQ_OK) return st;
  // 0 for arguments kvq_decode_attn rejects itself, below
  const size_t need = kvq_decode_workspace_size(desc, batch, num_q_heads, max_seq_len, num_splits);
  if (need > KVQ_STATIC_WORKSPACE_BYTES) return KVQ_ERR_WORKSPACE;
  return kvq_decode_attn(desc, cache, batch, num_q_heads, q, seq_lens, max_seq_len, num_splits,
                         softmax_scale, out, scratch, KVQ_STATIC_WORKSPACE_BYTES, dev_status,
                         stream);
}
