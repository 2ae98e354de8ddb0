// Dispatch of the chunk attention (kvq_chunk.cuh): the dequantize pass over
// every tile of every unit, then the attention kernel, one CTA per 256
// (query, head) rows of each unit, on the same stream.
#include "kvq_chunk.cuh"

namespace kvq {

int chunk_queries_per_cta(int gqa) { return gqa >= 1 && gqa <= kChunkRows ? kChunkRows / gqa : 0; }

size_t chunk_tile_bytes(int D) { return D == 128 ? ChunkTile<128>::bytes : ChunkTile<64>::bytes; }

namespace {
template <int D>
cudaError_t launch_attn(const ChunkParams& p, int units, cudaStream_t s) {
  static bool ready = false;  // shared-memory attribute, set once (single device)
  if (!ready) {
    const cudaError_t e =
        cudaFuncSetAttribute(chunk_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, ChunkSmem<D>::bytes);
    if (e != cudaSuccess) return e;
    ready = true;
  }
  const int blocks = (p.n + p.qpb - 1) / p.qpb;
  chunk_attn_kernel<D><<<dim3(blocks, units), kChunkCtaThreads, ChunkSmem<D>::bytes, s>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t chunk_attn_launch(int kb, int vb, int D, const ChunkParams& p, int units, int tiles, cudaStream_t s) {
  if (D != 64 && D != 128) return cudaErrorInvalidValue;
  ChunkDequant k{nullptr};
  switch (kb) {
    case 2: k = chunk_dequant_get_k2(vb, D); break;
    case 3: k = chunk_dequant_get_k3(vb, D); break;
    case 4: k = chunk_dequant_get_k4(vb, D); break;
    case 8: k = chunk_dequant_get_k8(vb, D); break;
    default: break;
  }
  if (!k.fn) return cudaErrorInvalidValue;
  k.fn<<<dim3(tiles, units), kDequantThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return D == 128 ? launch_attn<128>(p, units, s) : launch_attn<64>(p, units, s);
}

}  // namespace kvq
