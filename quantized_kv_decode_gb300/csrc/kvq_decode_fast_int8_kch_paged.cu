// Tensor-core decode kernel instantiations for INT8 axis-aware caches in the
// paged layout (the dense ones are in kvq_decode_fast_int8_kch.cu; K
// grouped per channel over blocks of g tokens; g a multiple of the 32-token
// tile, so that no tile straddles two blocks).
#include "kvq_decode_fast.cuh"

namespace kvq {

template <int D, int NG>
static cudaError_t by_gp_kch_paged(const DecodeParams& p, int gp, cudaStream_t s,
                                   bool* handled, int* occ) {
  *handled = true;
  switch (gp) {
    case 1: return fast::launch_fast_inst<8, D, NG, 1, false, true, false, true>(p, s, occ);
    case 2: return fast::launch_fast_inst<8, D, NG, 2, false, true, false, true>(p, s, occ);
    case 4: if constexpr (NG * 4 <= 16) return fast::launch_fast_inst<8, D, NG, 4, false, true, false, true>(p, s, occ);
            break;
    case 8: if constexpr (NG * 8 <= 16) return fast::launch_fast_inst<8, D, NG, 8, false, true, false, true>(p, s, occ);
            break;
  }
  *handled = false;
  return cudaSuccess;
}

cudaError_t launch_decode_fast_int8_kch_paged(const DecodeParams& p, int gp, cudaStream_t s,
                                              bool* handled, int* occ) {
  *handled = false;
  const int D = p.geom.D, NG = p.geom.ngroups;
  if (p.geom.g % fast::kTT) return cudaSuccess;
  if (D == 128 && NG == 4) return by_gp_kch_paged<128, 4>(p, gp, s, handled, occ);
  if (D == 128 && NG == 2) return by_gp_kch_paged<128, 2>(p, gp, s, handled, occ);
  if (D == 64 && NG == 2) return by_gp_kch_paged<64, 2>(p, gp, s, handled, occ);
  return cudaSuccess;
}

}  // namespace kvq
