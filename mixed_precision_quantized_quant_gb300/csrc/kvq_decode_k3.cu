// Decode-attention instantiations for 3-bit keys (all value widths,
// head_dim 64/128, up to 4 or 8 query heads per kv head).
#include "kvq_decode.cuh"
#include "kvq_kernels.h"

namespace kvq {

template <int VB, int D, int NT, int KM>
static DecodeKernel make() {
  DecodeKernel k;
  k.fn = decode_kernel<3, VB, D, NT, KM>;
  k.smem = 0;
  k.ctas_per_sm = 0;
  k.threads = 32 * decode_warps<3, VB, D, NT, KM>();
  return k;
}

DecodeKernel decode_get_k3(int vb, int D, int nt, int km) {
  DecodeKernel none{nullptr, 0, 0, 0};
  if (km != 0) return none;  // per-token keys are 2, 4 or 8 bits
#define E(VB)                                                                     \
  if (vb == VB) {                                                                 \
    if (D == 128) return nt == 1 ? make<VB, 128, 1, 0>() : make<VB, 128, 2, 0>(); \
    return nt == 1 ? make<VB, 64, 1, 0>() : make<VB, 64, 2, 0>();                 \
  }
  E(2) E(3) E(4) E(8)
#undef E
  return none;
}

}  // namespace kvq
