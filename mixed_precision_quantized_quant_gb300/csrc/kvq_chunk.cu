// Dispatch of the chunk-attention kernels (kvq_chunk.cuh): selects the
// (k_bits, v_bits, head_dim) instantiation, sets its shared-memory attribute
// once, and launches one CTA per 256 (query, head) rows of each unit.
#include "kvq_kernels.h"

namespace kvq {

namespace {
constexpr int kRowsPerCta = 256;
constexpr int kThreadsPerCta = 256;

int bits_index(int b) { return b == 2 ? 0 : b == 3 ? 1 : b == 4 ? 2 : b == 8 ? 3 : -1; }
}  // namespace

int chunk_queries_per_cta(int gqa) { return gqa >= 1 && gqa <= kRowsPerCta ? kRowsPerCta / gqa : 0; }

cudaError_t chunk_attn_launch(int kb, int vb, int D, const ChunkParams& p, int units, cudaStream_t s) {
  const int ik = bits_index(kb), iv = bits_index(vb);
  if (ik < 0 || iv < 0 || (D != 64 && D != 128)) return cudaErrorInvalidValue;
  ChunkKernel k{nullptr, 0};
  switch (kb) {
    case 2: k = chunk_get_k2(vb, D); break;
    case 3: k = chunk_get_k3(vb, D); break;
    case 4: k = chunk_get_k4(vb, D); break;
    default: k = chunk_get_k8(vb, D); break;
  }
  if (!k.fn) return cudaErrorInvalidValue;
  // shared-memory attribute, set once per instantiation (single device)
  static bool ready[4][4][2] = {};
  bool& r = ready[ik][iv][D == 128 ? 1 : 0];
  if (!r) {
    const cudaError_t e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem);
    if (e != cudaSuccess) return e;
    r = true;
  }
  const int blocks = (p.n + p.qpb - 1) / p.qpb;
  k.fn<<<dim3(blocks, units), kThreadsPerCta, k.smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
