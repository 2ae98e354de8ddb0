// Host-visible entry points of the CUDA kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"

namespace kvq {

// Fused quantize + pack + append, bit-width specialised.
cudaError_t append_dispatch(int kb, int vb, int D, const AppendParams& p, dim3 grid, int threads, size_t smem,
                            cudaStream_t s);
size_t append_smem_bytes(int kb, int vb, int D, int G, int rec_bytes);
// Threads of a CTA that quantizes key groups of G tokens.
int append_block_threads(int kb, int vb, int G);
// CTAs of the append kernel resident per SM at that block and shared-memory size (0 on error).
int append_ctas_per_sm(int kb, int vb, int D, int G, int threads, size_t smem);

// Decode attention, specialised on (k_bits, v_bits, head_dim, n-tiles).
typedef void (*decode_kernel_t)(DecodeParams);
struct DecodeKernel {
  decode_kernel_t fn;
  size_t smem;      // dynamic shared memory per CTA
  int ctas_per_sm;  // occupancy at that smem
  int threads;      // threads per CTA
};
// km: key mode (0 per channel over key groups, 1 per token).
// Returns fn == nullptr if the combination has no instantiation.
DecodeKernel decode_select(int kb, int vb, int D, int gqa, int km);
size_t decode_smem_bytes(int kb, int vb, int D, int nt, int km, int warps);

// Causal multi-query attention over the quantized cache: a dequantize pass
// (specialised on (k_bits, v_bits, head_dim)) writes every 64-token tile of
// every unit into the workspace, then the attention kernel (specialised on
// head_dim; tensor-core MMAs with accumulators in tensor memory) reads them.
struct ChunkDequant {
  void (*fn)(ChunkParams);
};
ChunkDequant chunk_dequant_get_k2(int vb, int D);
ChunkDequant chunk_dequant_get_k3(int vb, int D);
ChunkDequant chunk_dequant_get_k4(int vb, int D);
ChunkDequant chunk_dequant_get_k8(int vb, int D);
// Bytes of one dequantized tile in the workspace.
size_t chunk_tile_bytes(int D);
// Both launches; `tiles` = the unit's tiles at the current length.
cudaError_t chunk_attn_launch(int kb, int vb, int D, const ChunkParams& p, int units, int tiles, cudaStream_t s);
// Queries of the n newest tokens that one CTA serves (256 (query, head) rows).
int chunk_queries_per_cta(int gqa);

}  // namespace kvq
