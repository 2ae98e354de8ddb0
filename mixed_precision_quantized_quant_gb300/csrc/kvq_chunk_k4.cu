// Chunk-attention instantiations for 4-bit keys (all value widths, head_dim 64/128).
#include "kvq_chunk.cuh"

namespace kvq {

ChunkKernel chunk_get_k4(int vb, int D) {
#define E(VB) \
  if (vb == VB) return D == 128 ? chunk_make<4, VB, 128>() : chunk_make<4, VB, 64>();
  E(2) E(3) E(4) E(8)
#undef E
  return ChunkKernel{nullptr, 0};
}

}  // namespace kvq
