// Maps a layer's (k_bits, v_bits, head_dim, query heads per kv head) to its
// decode-attention instantiation, its shared-memory size and occupancy.
#include "kvq_decode.cuh"
#include "kvq_kernels.h"

namespace kvq {

DecodeKernel decode_get_k2(int vb, int D, int nt, int km);
DecodeKernel decode_get_k3(int vb, int D, int nt, int km);
DecodeKernel decode_get_k4(int vb, int D, int nt, int km);
DecodeKernel decode_get_k8(int vb, int D, int nt, int km);

static int words(int D, int b) { return b == 3 ? (D + 10) / 11 : D * b / 32; }

size_t decode_smem_bytes(int kb, int vb, int D, int nt, int km, int warps) {
  const int cq = slice_bytes(D, words(D, kb), words(D, vb), km);
  return static_cast<size_t>(decode_smem_layout(D, nt, cq, warps).total);
}

DecodeKernel decode_select(int kb, int vb, int D, int gqa, int km) {
  DecodeKernel k{nullptr, 0, 0, 0};
  if (gqa < 1 || gqa > 8) return k;
  const int nt = gqa <= 4 ? 1 : 2;
  if (kb == 2) k = decode_get_k2(vb, D, nt, km);
  else if (kb == 3) k = decode_get_k3(vb, D, nt, km);
  else if (kb == 4) k = decode_get_k4(vb, D, nt, km);
  else if (kb == 8) k = decode_get_k8(vb, D, nt, km);
  if (!k.fn) return k;
  k.smem = decode_smem_bytes(kb, vb, D, nt, km, k.threads / 32);
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
