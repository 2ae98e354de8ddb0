// Maps a layer's (k_bits, v_bits, head_dim, query heads per kv head) to its
// decode-attention instantiation, its shared-memory size and occupancy.
#include "kvq_decode.cuh"
#include "kvq_kernels.h"

namespace kvq {

DecodeKernel decode_get_k2(int vb, int D, int nt);
DecodeKernel decode_get_k3(int vb, int D, int nt);
DecodeKernel decode_get_k4(int vb, int D, int nt);
DecodeKernel decode_get_k8(int vb, int D, int nt);

size_t decode_smem_bytes(int D, int nt, int G, int rec_bytes, int warps) {
  return static_cast<size_t>(decode_smem_layout(D, nt, G, rec_bytes, warps).total);
}

DecodeKernel decode_select(int kb, int vb, int D, int gqa, int G, int rec_bytes) {
  DecodeKernel k{nullptr, 0, 0, 0};
  if (gqa < 1 || gqa > 8) return k;
  const int nt = gqa <= 4 ? 1 : 2;
  if (kb == 2) k = decode_get_k2(vb, D, nt);
  else if (kb == 3) k = decode_get_k3(vb, D, nt);
  else if (kb == 4) k = decode_get_k4(vb, D, nt);
  else if (kb == 8) k = decode_get_k8(vb, D, nt);
  if (!k.fn) return k;
  k.smem = decode_smem_bytes(D, nt, G, rec_bytes, k.threads / 32);
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(k.fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(k.smem)) != cudaSuccess) {
    k.fn = nullptr;
    return k;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, reinterpret_cast<const void*>(k.fn), k.threads,
                                                    k.smem) != cudaSuccess || occ < 1) {
    k.fn = nullptr;
    return k;
  }
  k.ctas_per_sm = occ;
  return k;
}

}  // namespace kvq
