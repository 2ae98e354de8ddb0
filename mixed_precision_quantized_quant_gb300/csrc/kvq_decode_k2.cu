// Decode-attention instantiations for 2-bit keys (all value widths,
// head_dim 64/128, up to 4 or 8 query heads per kv head).
#include "kvq_decode.cuh"
#include "kvq_kernels.h"

namespace kvq {

template <int VB, int D, int NT, int KM>
static DecodeKernel make() {
  DecodeKernel k;
  k.fn = decode_kernel<2, VB, D, NT, KM>;
  k.smem = 0;
  k.ctas_per_sm = 0;
  k.threads = 32 * decode_warps<2, VB, D, NT, KM>();
  return k;
}

DecodeKernel decode_get_k2(int vb, int D, int nt, int km) {
  DecodeKernel none{nullptr, 0, 0, 0};
#define E(VB)                                                                         \
  if (vb == VB) {                                                                     \
    if (km == 0) {                                                                    \
      if (D == 128) return nt == 1 ? make<VB, 128, 1, 0>() : make<VB, 128, 2, 0>();   \
      return nt == 1 ? make<VB, 64, 1, 0>() : make<VB, 64, 2, 0>();                   \
    }                                                                                 \
    if (D == 128) return nt == 1 ? make<VB, 128, 1, 1>() : make<VB, 128, 2, 1>();     \
    return nt == 1 ? make<VB, 64, 1, 1>() : make<VB, 64, 2, 1>();                     \
  }
  E(2) E(3) E(4) E(8)
#undef E
  return none;
}

}  // namespace kvq
