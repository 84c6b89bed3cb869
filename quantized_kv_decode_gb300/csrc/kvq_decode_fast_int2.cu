// Tensor-core decode kernel instantiations for INT2 caches (four codes per
// byte), asymmetric and symmetric, head_dim 128.  A 16-byte chunk holds 64
// channels; chunks that span several groups (g16, g32) need every (group,
// head) column in one V-mma n-tile, so those group sizes take up to 8 / NG
// query heads per KV head.
#include "kvq_decode_fast.cuh"

namespace kvq {

template <int NG, bool SYM>
static cudaError_t by_gp2(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                          int* occ) {
  *handled = true;
  switch (gp) {
    case 1: return fast::launch_fast_inst<2, 128, NG, 1, SYM>(p, s, occ);
    case 2: if constexpr (NG * 2 <= 8) return fast::launch_fast_inst<2, 128, NG, 2, SYM>(p, s, occ);
            break;
    case 4: if constexpr (NG == 2) return fast::launch_fast_inst<2, 128, NG, 4, SYM>(p, s, occ);
            break;
    case 8: if constexpr (NG == 2) return fast::launch_fast_inst<2, 128, NG, 8, SYM>(p, s, occ);
            break;
  }
  *handled = false;
  return cudaSuccess;
}

cudaError_t launch_decode_fast_int2(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                                    int* occ) {
  *handled = false;
  if (p.geom.D != 128 || p.geom.kch) return cudaSuccess;
  const int NG = p.geom.ngroups;
  if (p.geom.sym) {
    if (NG == 2) return by_gp2<2, true>(p, gp, s, handled, occ);
    if (NG == 4) return by_gp2<4, true>(p, gp, s, handled, occ);
    if (NG == 8) return by_gp2<8, true>(p, gp, s, handled, occ);
  } else {
    if (NG == 2) return by_gp2<2, false>(p, gp, s, handled, occ);
    if (NG == 4) return by_gp2<4, false>(p, gp, s, handled, occ);
    if (NG == 8) return by_gp2<8, false>(p, gp, s, handled, occ);
  }
  return cudaSuccess;
}

}  // namespace kvq
