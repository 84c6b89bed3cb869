// Decode over fp16 caches: the tensor-core kernel (kvq_decode_f16.cuh) for
// head_dim 64 / 128 with at most 8 query heads per KV head, the CUDA-core
// kernel for the other shapes.
#include "kvq_decode_cc.cuh"
#include "kvq_decode_f16.cuh"

namespace kvq {

cudaError_t launch_decode_cc_b16(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm) {
  bool handled = false;
  const cudaError_t e = f16::launch(p, stream, ctas_per_sm, &handled);
  if (handled) return e;
  return cc::launch_cc_bits<16>(p, stream, ctas_per_sm);
}

}  // namespace kvq
