// Fused quantize + pack + append for one layer of the mixed-precision KV cache.
//
// One CTA (4 warps) per (unit, job); a unit is one (batch, kv head).  A job is
// either one key group to quantize ("flush") or a chunk of new tokens to copy
// into the FP16 residual ring.  Keys are quantized per channel over the G
// tokens of a group, values per token, with
//   scale = (max - min)/(2^b - 1) in fp32, stored fp16; zero = min;
//   code  = clamp(rint((x - min) / scale), 0, 2^b - 1)
// ("KVTuner ...", section A3 quantizer; "KVmix ...", 关键设计 2; "LLM 量化精读笔记
// · 08 ...", sections 6.1-6.2).  The division is the IEEE fp32 one: a
// reciprocal estimate decides the code unless the quotient lies within 2^-14
// of a rounding boundary, where the correctly rounded __fdiv_rn decides.
//
// Per-channel and per-token min/max use warp shuffles; packed codes are
// assembled in shared memory and leave as one bulk (TMA) store per group.
#include "kvq_device.cuh"
#include "kvq_kernels.h"

namespace kvq {
namespace {

template <int B>
struct BitsT {
  static constexpr int kQmax = (1 << B) - 1;
};

__host__ __device__ constexpr int words_per_row(int d, int b) { return b == 3 ? (d + 10) / 11 : d * b / 32; }

// code = clamp(rint(a / s), 0, qmax) with a = x - min already rounded to fp32;
// s > 0 is the fp32 value of the stored scale, r = 1/s (rounded).
__device__ __forceinline__ uint32_t code_of(float a, float s, float r, float qmax) {
  const float y = __fmul_rn(a, r);
  float q = rintf(y);
  const float dist = fabsf(__fsub_rn(y, q));
  if (fabsf(dist - 0.5f) <= 6.103515625e-05f) {  // 2^-14: decide with the exact quotient
    q = rintf(__fdiv_rn(a, s));
  }
  q = fminf(fmaxf(q, 0.0f), qmax);
  return static_cast<uint32_t>(q);
}

struct Scale {
  float mn;   // zero (fp16 value, exact in fp32)
  float s;    // stored fp16 scale as fp32
  float r;    // 1/s
  float qmax;
  __half s16, z16;
};

template <int B>
__device__ __forceinline__ Scale make_scale(__half mn, __half mx, bool slot10) {
  Scale sc;
  const float fmn = __half2float(mn), fmx = __half2float(mx);
  const float s32 = __fdiv_rn(__fsub_rn(fmx, fmn), static_cast<float>(BitsT<B>::kQmax));
  sc.s16 = __float2half_rn(s32);
  sc.z16 = mn;
  sc.mn = fmn;
  float s = __half2float(sc.s16);
  sc.qmax = static_cast<float>(BitsT<B>::kQmax);
  if (B == 3 && slot10) {  // 2-bit field of an 11-field word: s2 = (s*7)/3
    s = __fdiv_rn(__fmul_rn(s, 7.0f), 3.0f);
    sc.qmax = 3.0f;
  }
  sc.s = s;
  sc.r = (s > 0.0f) ? __frcp_rn(s) : 0.0f;
  return sc;
}

__device__ __forceinline__ uint32_t quant(float x, const Scale& sc) {
  if (!(sc.s > 0.0f)) return 0u;
  return code_of(__fsub_rn(x, sc.mn), sc.s, sc.r, sc.qmax);
}

__device__ __forceinline__ void h8(const uint4& v, __half (&h)[8]) {
  const __half2* p = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = __low2half(p[i]);
    h[2 * i + 1] = __high2half(p[i]);
  }
}

// Packs 8 consecutive codes (channels c0..c0+7, c0 % 8 == 0) of bit width B.
// Returns the low/high word (B == 8: two words; B == 4: one; B == 2: 16 bits).
template <int B>
__device__ __forceinline__ void pack8(const uint32_t (&c)[8], uint32_t& w0, uint32_t& w1) {
  w0 = 0;
  w1 = 0;
  if (B == 8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) w0 |= c[j] << (8 * j);
#pragma unroll
    for (int j = 0; j < 4; ++j) w1 |= c[4 + j] << (8 * j);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) w0 |= c[j] << (B * j);
  }
}

// Row chunk address of token i (absolute position) of unit u: the FP16 ring
// if the token was appended before this call, else the caller's input.
__device__ __forceinline__ const uint4* src_chunk(const AppendParams& p, const __half* ring, const __half* in,
                                                  int u, int64_t i, int64_t T, int chunk, int D) {
  if (i < T) {
    const int slot = static_cast<int>(i % p.R);
    const int phys = chunk ^ (slot & 7);
    return reinterpret_cast<const uint4*>(ring + u * p.res_stride + static_cast<int64_t>(slot) * D) + phys;
  }
  const int64_t j = i - T;
  return reinterpret_cast<const uint4*>(in + (static_cast<int64_t>(u) * p.n + j) * D) + chunk;
}

template <int KB, int VB, int D>
__device__ void quantize_group(const AppendParams& p, int u, int64_t grp, int64_t T, uint8_t* smem) {
  constexpr int WK = words_per_row(D, KB);
  constexpr int WV = words_per_row(D, VB);
  const int G = p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* rec = smem;
  uint32_t* kc = reinterpret_cast<uint32_t*>(rec);
  uint32_t* vc = kc + G * WK;
  __half* ks = reinterpret_cast<__half*>(vc + G * WV);
  __half* kz = ks + D;
  __half2* vsz = reinterpret_cast<__half2*>(kz + D);
  uint8_t* bytes = rec + p.rec_bytes;  // 3-bit staging: [G][D] codes
  const int64_t t0 = grp * G;

  // ---------------- keys: per channel over the group's G tokens
  {
    constexpr int CW = D / 4;          // channels per warp
    constexpr int LPR = CW / 8;        // lanes per token row
    constexpr int RPL = 32 / LPR;      // token rows per warp-load
    constexpr int NLMAX = 128 / RPL;   // loads for the largest group
    const int r = lane / LPR, cs = lane % LPR;
    const int cb = warp * CW + cs * 8;  // first of this lane's 8 channels
    const int nl = G / RPL;
    uint4 x[NLMAX];
    __half2 mn[4], mx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      mn[k] = __float2half2_rn(65504.f);
      mx[k] = __float2half2_rn(-65504.f);
    }
#pragma unroll
    for (int it = 0; it < NLMAX; ++it) {
      if (it < nl) {
        const int64_t i = t0 + it * RPL + r;
        x[it] = *src_chunk(p, p.res_k, p.K, u, i, T, cb / 8, D);
        const __half2* h = reinterpret_cast<const __half2*>(&x[it]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          mn[k] = __hmin2(mn[k], h[k]);
          mx[k] = __hmax2(mx[k], h[k]);
        }
      }
    }
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t a = __shfl_xor_sync(0xffffffffu, h2_as_u32(mn[k]), off);
        const uint32_t b = __shfl_xor_sync(0xffffffffu, h2_as_u32(mx[k]), off);
        mn[k] = __hmin2(mn[k], u32_as_h2(a));
        mx[k] = __hmax2(mx[k], u32_as_h2(b));
      }
    }
    Scale sc[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      sc[2 * k] = make_scale<KB>(__low2half(mn[k]), __low2half(mx[k]), (cb + 2 * k) % 11 == 10);
      sc[2 * k + 1] = make_scale<KB>(__high2half(mn[k]), __high2half(mx[k]), (cb + 2 * k + 1) % 11 == 10);
    }
    if (r == 0) {
      __half s8[8], z8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        s8[k] = sc[k].s16;
        z8[k] = sc[k].z16;
      }
      *reinterpret_cast<uint4*>(ks + cb) = *reinterpret_cast<uint4*>(s8);
      *reinterpret_cast<uint4*>(kz + cb) = *reinterpret_cast<uint4*>(z8);
    }
#pragma unroll
    for (int it = 0; it < NLMAX; ++it) {
      if (it < nl) {
        const int t = it * RPL + r;
        __half h[8];
        h8(x[it], h);
        uint32_t c[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] = quant(__half2float(h[k]), sc[k]);
        if (KB == 3) {
          uint32_t lo = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
          uint32_t hi = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
          *reinterpret_cast<uint2*>(bytes + t * D + cb) = make_uint2(lo, hi);
        } else {
          uint32_t w0, w1;
          pack8<KB>(c, w0, w1);
          if (KB == 8) {
            *reinterpret_cast<uint2*>(kc + t * WK + cb / 4) = make_uint2(w0, w1);
          } else if (KB == 4) {
            kc[t * WK + cb / 8] = w0;
          } else {  // KB == 2: two lanes form one word
            const uint32_t other = __shfl_xor_sync(0xffffffffu, w0, 1);
            if ((cs & 1) == 0) kc[t * WK + cb / 16] = w0 | (other << 16);
          }
        }
      }
    }
  }

  // ---------------- values: per token over its D channels
  {
    constexpr int TPL = D / 8;         // lanes per token
    constexpr int TPW = 32 / TPL;      // tokens per warp-load
    const int sub = lane / TPL, cs = lane % TPL;
    const int cb = cs * 8;
    for (int t = (warp * TPW) + sub; t < G; t += kWarps * TPW) {
      const int64_t i = t0 + t;
      const uint4 x = *src_chunk(p, p.res_v, p.V, u, i, T, cs, D);
      const __half2* h2 = reinterpret_cast<const __half2*>(&x);
      __half2 mn2 = __hmin2(__hmin2(h2[0], h2[1]), __hmin2(h2[2], h2[3]));
      __half2 mx2 = __hmax2(__hmax2(h2[0], h2[1]), __hmax2(h2[2], h2[3]));
      __half mn = __hmin(__low2half(mn2), __high2half(mn2));
      __half mx = __hmax(__low2half(mx2), __high2half(mx2));
#pragma unroll
      for (int off = 1; off < TPL; off <<= 1) {
        const __half a = __ushort_as_half(
            static_cast<unsigned short>(__shfl_xor_sync(0xffffffffu, __half_as_ushort(mn), off)));
        const __half b = __ushort_as_half(
            static_cast<unsigned short>(__shfl_xor_sync(0xffffffffu, __half_as_ushort(mx), off)));
        mn = __hmin(mn, a);
        mx = __hmax(mx, b);
      }
      const Scale s3 = make_scale<VB>(mn, mx, false);
      Scale s2 = s3;
      if (VB == 3) s2 = make_scale<VB>(mn, mx, true);
      __half h[8];
      h8(x, h);
      uint32_t c[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const bool two = (VB == 3) && ((cb + k) % 11 == 10);
        c[k] = quant(__half2float(h[k]), two ? s2 : s3);
      }
      if (cs == 0) vsz[t] = __halves2half2(s3.s16, s3.z16);
      if (VB == 3) {
        uint32_t lo = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
        uint32_t hi = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
        *reinterpret_cast<uint2*>(bytes + G * D + t * D + cb) = make_uint2(lo, hi);
      } else {
        uint32_t w0, w1;
        pack8<VB>(c, w0, w1);
        if (VB == 8) {
          *reinterpret_cast<uint2*>(vc + t * WV + cb / 4) = make_uint2(w0, w1);
        } else if (VB == 4) {
          vc[t * WV + cb / 8] = w0;
        } else {
          const uint32_t other = __shfl_xor_sync(0xffffffffu, w0, 1);
          if ((cs & 1) == 0) vc[t * WV + cb / 16] = w0 | (other << 16);
        }
      }
    }
  }

  // ---------------- 3-bit words: ten 3-bit fields and one 2-bit field
  if (KB == 3 || VB == 3) {
    __syncthreads();
    if (KB == 3) {
      for (int idx = tid; idx < G * WK; idx += kThreads) {
        const int t = idx / WK, w = idx % WK;
        uint32_t word = 0;
        for (int j = 0; j < 11; ++j) {
          const int c = 11 * w + j;
          if (c < D) word |= static_cast<uint32_t>(bytes[t * D + c]) << (j == 10 ? 30 : 3 * j);
        }
        kc[idx] = word;
      }
    }
    if (VB == 3) {
      for (int idx = tid; idx < G * WV; idx += kThreads) {
        const int t = idx / WV, w = idx % WV;
        uint32_t word = 0;
        for (int j = 0; j < 11; ++j) {
          const int c = 11 * w + j;
          if (c < D) word |= static_cast<uint32_t>(bytes[G * D + t * D + c]) << (j == 10 ? 30 : 3 * j);
        }
        vc[idx] = word;
      }
    }
  }

  // ---------------- one bulk store of the finished record
  __syncthreads();
  if (tid == 0) {
    fence_proxy_async_smem();
    uint8_t* dst = p.records + static_cast<int64_t>(u) * p.unit_rec_stride + grp * p.rec_bytes;
    bulk_s2g(dst, rec, static_cast<uint32_t>(p.rec_bytes));
    bulk_commit();
    bulk_wait_all();
  }
  __syncthreads();
}

// Copy new tokens [lo, hi) (absolute positions, all from this call's input)
// into the unit's FP16 rings, 16-byte chunks swizzled by slot.
template <int D>
__device__ void write_residual(const AppendParams& p, int u, int64_t lo, int64_t hi, int64_t T) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const int64_t n = hi - lo;
  for (int64_t idx = threadIdx.x; idx < n * 2 * CH; idx += kThreads) {
    const int64_t tok = lo + idx / (2 * CH);
    const int rem = static_cast<int>(idx % (2 * CH));
    const int which = rem / CH, c = rem % CH;
    const __half* in = which ? p.V : p.K;
    __half* ring = which ? p.res_v : p.res_k;
    const uint4 v = reinterpret_cast<const uint4*>(in + (static_cast<int64_t>(u) * p.n + (tok - T)) * D)[c];
    const int slot = static_cast<int>(tok % p.R);
    reinterpret_cast<uint4*>(ring + u * p.res_stride + static_cast<int64_t>(slot) * D)[c ^ (slot & 7)] = v;
  }
}

template <int KB, int VB, int D>
__global__ void __launch_bounds__(kThreads) append_kernel(AppendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int u = blockIdx.y;
  const int64_t T = __ldcg(p.tokens);
  const int64_t nq0 = quantized_after(T, p.R, p.G);
  const int64_t nq1 = quantized_after(T + p.n, p.R, p.G);

  if (p.mode & kFlush) {
    const int64_t grp = nq0 / p.G + blockIdx.x;
    if (grp < nq1 / p.G) quantize_group<KB, VB, D>(p, u, grp, T, smem);
  }
  if (p.mode & kResidual) {
    // tokens that stay in the window after this call
    const int64_t first = (T > nq1) ? T : nq1;
    const int64_t last = T + p.n;
    if (p.mode & kFlush) {  // fused single-CTA-per-unit launch writes them all
      if (first < last) write_residual<D>(p, u, first, last, T);
    } else {
      const int64_t per = 16;
      const int64_t lo = first + static_cast<int64_t>(blockIdx.x) * per;
      const int64_t hi = (lo + per < last) ? lo + per : last;
      if (lo < hi) write_residual<D>(p, u, lo, hi, T);
    }
  }
  if (p.mode & kUpdateState) {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int prev = atomicAdd(p.done_ctr, 1);
      if (prev == p.ctas - 1) {
        *p.tokens = static_cast<int32_t>(T + p.n);
        *p.done_ctr = 0;
        __threadfence();
      }
    }
  }
}

}  // namespace

template <int KB, int VB, int D>
static cudaError_t launch_append(const AppendParams& p, dim3 grid, size_t smem, cudaStream_t s) {
  auto k = append_kernel<KB, VB, D>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

#define KVQ_APPEND_ENTRY(KB, VB)                                                     \
  case (KB * 16 + VB):                                                              \
    return D == 128 ? launch_append<KB, VB, 128>(p, grid, smem, s)                  \
                    : launch_append<KB, VB, 64>(p, grid, smem, s);

cudaError_t append_dispatch(int kb, int vb, int D, const AppendParams& p, dim3 grid, size_t smem,
                            cudaStream_t s) {
  switch (kb * 16 + vb) {
    KVQ_APPEND_ENTRY(2, 2) KVQ_APPEND_ENTRY(2, 3) KVQ_APPEND_ENTRY(2, 4) KVQ_APPEND_ENTRY(2, 8)
    KVQ_APPEND_ENTRY(3, 2) KVQ_APPEND_ENTRY(3, 3) KVQ_APPEND_ENTRY(3, 4) KVQ_APPEND_ENTRY(3, 8)
    KVQ_APPEND_ENTRY(4, 2) KVQ_APPEND_ENTRY(4, 3) KVQ_APPEND_ENTRY(4, 4) KVQ_APPEND_ENTRY(4, 8)
    KVQ_APPEND_ENTRY(8, 2) KVQ_APPEND_ENTRY(8, 3) KVQ_APPEND_ENTRY(8, 4) KVQ_APPEND_ENTRY(8, 8)
    default:
      return cudaErrorInvalidValue;
  }
}

size_t append_smem_bytes(int kb, int vb, int D, int G, int rec_bytes) {
  size_t b = static_cast<size_t>(rec_bytes);
  if (kb == 3 || vb == 3) b += static_cast<size_t>(2) * G * D;
  return (b + 127) / 128 * 128;
}

}  // namespace kvq
