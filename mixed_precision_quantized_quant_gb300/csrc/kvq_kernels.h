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
int append_block_threads(int G);
// CTAs of the append kernel resident per SM at that block and shared-memory size (0 on error).
int append_ctas_per_sm(int kb, int vb, int D, int threads, size_t smem);

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

}  // namespace kvq
