// Tensor-core decode kernel instantiations for NF4 caches: 4-bit codes that
// index the sixteen normal-quantile levels, one absmax scale per group, no
// zero arrays.  The codes become fp16 levels by a byte-permute lookup.
#include "kvq_decode_fast.cuh"

namespace kvq {

template <int D, int NG>
static cudaError_t by_gp_nf4(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                             int* occ) {
  *handled = true;
  switch (gp) {
    case 1: return fast::launch_fast_inst<4, D, NG, 1, true, false, true>(p, s, occ);
    case 2: return fast::launch_fast_inst<4, D, NG, 2, true, false, true>(p, s, occ);
    case 4: return fast::launch_fast_inst<4, D, NG, 4, true, false, true>(p, s, occ);
    case 8: if constexpr (NG * 8 <= 16) return fast::launch_fast_inst<4, D, NG, 8, true, false, true>(p, s, occ);
            break;
  }
  *handled = false;
  return cudaSuccess;
}

cudaError_t launch_decode_fast_nf4(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                                   int* occ) {
  *handled = false;
  const int D = p.geom.D, NG = p.geom.ngroups;
  if (D == 128 && NG == 2) return by_gp_nf4<128, 2>(p, gp, s, handled, occ);
  if (D == 128 && NG == 4) return by_gp_nf4<128, 4>(p, gp, s, handled, occ);
  if (D == 64 && NG == 2) return by_gp_nf4<64, 2>(p, gp, s, handled, occ);
  return cudaSuccess;
}

}  // namespace kvq
