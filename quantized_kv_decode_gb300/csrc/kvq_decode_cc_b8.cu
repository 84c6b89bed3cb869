// CUDA-core decode kernel instantiations for 8-bit codes (16: fp16 caches).
#include "kvq_decode_cc.cuh"

namespace kvq {

cudaError_t launch_decode_cc_b8(const DecodeParams& p, cudaStream_t stream, int* ctas_per_sm) {
  return cc::launch_cc_bits<8>(p, stream, ctas_per_sm);
}

}  // namespace kvq
