// Tensor-core decode kernel instantiations for INT8 caches with asymmetric codes
// (the symmetric ones are in kvq_decode_fast_int8_sym.cu).
#include "kvq_decode_fast.cuh"

namespace kvq {

template <int D, int NG>
static cudaError_t by_gp8(const DecodeParams& p, int gp, cudaStream_t s, bool* handled,
                          int* occ) {
  constexpr bool SYM = false;
  *handled = true;
  switch (gp) {
    case 1: return fast::launch_fast_inst<8, D, NG, 1, SYM>(p, s, occ);
    case 2: return fast::launch_fast_inst<8, D, NG, 2, SYM>(p, s, occ);
    case 4: if constexpr (NG * 4 <= 16) return fast::launch_fast_inst<8, D, NG, 4, SYM>(p, s, occ);
            break;
    case 8: if constexpr (NG * 8 <= 16) return fast::launch_fast_inst<8, D, NG, 8, SYM>(p, s, occ);
            break;
  }
  *handled = false;
  return cudaSuccess;
}

cudaError_t launch_decode_fast_int8(const DecodeParams& p, int gp, cudaStream_t s,
                                    bool* handled, int* occ) {
  *handled = false;
  if (p.geom.sym) return launch_decode_fast_int8_sym(p, gp, s, handled, occ);
  if (p.geom.kch)
    return p.geom.layout == KVQ_DENSE ? launch_decode_fast_int8_kch(p, gp, s, handled, occ)
                                      : launch_decode_fast_int8_kch_paged(p, gp, s, handled, occ);
  const int D = p.geom.D, NG = p.geom.ngroups;
  if (D == 128 && NG == 2) return by_gp8<128, 2>(p, gp, s, handled, occ);
  if (D == 128 && NG == 4) return by_gp8<128, 4>(p, gp, s, handled, occ);
  if (D == 128 && NG == 8) return by_gp8<128, 8>(p, gp, s, handled, occ);
  if (D == 64 && NG == 2) return by_gp8<64, 2>(p, gp, s, handled, occ);
  if (D == 64 && NG == 4) return by_gp8<64, 4>(p, gp, s, handled, occ);
  return cudaSuccess;
}

}  // namespace kvq
