// Dequantize-pass instantiations of the chunk attention for 4-bit keys
// (all value widths, head_dim 64/128).
#include "kvq_chunk.cuh"

namespace kvq {

ChunkDequant chunk_dequant_get_k4(int vb, int D) {
#define E(VB) \
  if (vb == VB) return D == 128 ? chunk_dequant_make<4, VB, 128>() : chunk_dequant_make<4, VB, 64>();
  E(2) E(3) E(4) E(8)
#undef E
  return ChunkDequant{nullptr};
}

}  // namespace kvq
