// Fused quantize + pack + append for one layer of the mixed-precision KV cache.
//
// A unit is one (batch, kv head).  Key groups to quantize ("flush jobs") are
// spread over persistent CTAs of 4*G threads: each CTA stages the K and V rows of
// its next group in shared memory with bulk (TMA) copies while it quantizes
// the current one.  New tokens that stay in the FP16 residual window are
// copied into the unit's ring by the same launch (one token per unit in a
// decode step) or by a second launch in 16-token chunks (prefill).  Keys are quantized per channel over the G
// tokens of a group, values per token, with
//   scale = (max - min)/(2^b - 1) in fp32, stored fp16; zero = min;
//   code  = clamp(rint((x - min) / scale), 0, 2^b - 1)
// ("KVTuner ...", section A3 quantizer; "KVmix ...", 关键设计 2; "LLM 量化精读笔记
// · 08 ...", sections 6.1-6.2).  The division is the IEEE fp32 one: a
// reciprocal estimate decides the code unless the product lies near a
// rounding boundary (kNearHalf states the band and why it suffices), where
// the correctly rounded __fdiv_rn decides.
//
// Per-channel min/max runs over the staged rows, per-token min/max uses warp
// shuffles; each scale is computed once, by one thread; packed codes are
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
  // 1/s only steers the fast path of the code computation: kNearHalf's band
  // covers a reciprocal with relative error up to 2^-22
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  sc.r = (s > 0.0f) ? r : 0.0f;
  return sc;
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

// Shared-memory layout of the flush path.
struct AppendSmem {
  int tile;  // bytes of one staged [G][D] fp16 tile
  int off_stage1, off_rec, off_ksc, off_kp, off_vsc, off_vr2, off_kmn, off_kmx, off_vpart, off_kpt, off_ksct,
      off_bars, total;
};

// Flush CTAs run 4*G threads, each owning one 16-byte chunk of D/32 rows, with
// two stages; "wide" CTAs (G = 128 without 3-bit codes) run 2*G threads, each
// owning one chunk of D/16 rows, with one stage that is refilled as soon as
// every thread holds its rows in registers, so that two CTAs fit an SM instead
// of one and cover each other's barrier waits.  (At G = 64 the same form, four
// 128-thread CTAs per SM instead of two of 256, measured no faster.)
__host__ __device__ constexpr bool append_wide(int KB, int VB, int G) { return G == 128 && KB != 3 && VB != 3; }
__host__ __device__ constexpr int append_threads(int G, bool wide) { return (wide ? 2 : 4) * G; }

__host__ __device__ inline AppendSmem append_smem_layout(int D, int G, int rec_bytes, bool wide) {
  AppendSmem a;
  a.tile = G * D * 2;
  const int warps = append_threads(G, wide) / 32;
  int off = 2 * a.tile;  // stage 0 at offset 0: K tile, then V tile
  a.off_stage1 = off;
  if (!wide) off += 2 * a.tile;
  a.off_rec = off;
  off += (rec_bytes + 127) / 128 * 128;
  a.off_ksc = off;
  off += D * 16;  // per channel {min, s, 1/s, qmax}, channel 8c + k at k*(D/8) + c
  a.off_kp = off;
  off += D * 8;   // per channel min and 1/s as pairs: {min[8c+2j], min[8c+2j+1]} at j*(D/8) + c,
                  // then the same for 1/s at D/2 + j*(D/8) + c (8 bytes each)
  a.off_vsc = off;
  off += G * 16;  // per token {min, s, 1/s, s2}
  a.off_vr2 = off;
  off += G * 4;   // per token 1/s2 (3-bit values)
  a.off_kmn = off;
  off += warps * D * 2;  // per warp, per channel: min over the warp's rows
  a.off_kmx = off;
  off += warps * D * 2;  // ... and max
  a.off_vpart = off;
  off += G * 4;   // per token {min, -max}
  a.off_kpt = off;
  off += G * 4;   // per-token keys: per token {min, -max}
  a.off_ksct = off;
  off += G * 16;  // per-token keys: per token {min, s, 1/s, qmax}
  a.off_bars = off;
  off += 16;
  a.total = off;
  return a;
}

// The band of the fast path, stated once.  It computes y = fl((x - min) * r)
// with r = rcp.approx(s); the code must equal rint(fl((x - min) / s)).
//   * r = (1/s)(1 + e1) with |e1| <= 2^-22 (the PTX ISA gives rcp.approx.f32
//     a 1-ulp bound, about 2^-23; the argument only needs twice that);
//   * the product's rounding adds |e2| <= 2^-24, so |y - a/s| <= (a/s) *
//     (2^-22 + 2^-24 + 2^-46), a = x - min;
//   * the IEEE quotient is within 2^-24 * (a/s) of a/s;
//   * a/s <= 1.5 * 255 < 383 (the fp16 scale is at least s32 / 1.5, and
//     far closer for normal scales).
// So |y - fl(a/s)| <= 383 * (2^-22 + 2^-23 + 2^-46) < 1.37e-4 < 2^-12.  If y
// is at least 2^-12 away from every rounding boundary k + 1/2, the IEEE
// quotient lies on the same side of it and both round to the same integer;
// every y inside the band is redone with the IEEE division.  (fp32 resolves
// the band: below 512 the spacing of y is at most 2^-15.)
constexpr float kNearHalf = 0.5f - 2.44140625e-04f;  // within 2^-12 of a boundary: exact path

// code = min(rint((x - min) / s), qmax) with IEEE fp32 subtraction and
// division: the product with 1/s decides outside kNearHalf's band, the
// correctly rounded quotient inside it.  x >= min always, so no lower clamp.
// sc = {min, s, 1/s, qmax}; s == 0 carries 1/s == 0 and gives code 0.
__device__ __forceinline__ uint32_t quant_fast(float x, const float4& sc) {
  const float a = __fsub_rn(x, sc.x);
  const float y = __fmul_rn(a, sc.z);
  float q = rintf(y);
  if (fabsf(__fsub_rn(y, q)) >= kNearHalf && sc.z > 0.0f) q = rintf(__fdiv_rn(a, sc.y));
  return static_cast<uint32_t>(fminf(q, sc.w));
}

// The rare exact path of quant8, kept out of line so the common path stays
// compact.  Scales come from the shared-memory table (element k at
// tab[k * stride]; qmax from the table when qm < 0); the eight codes return
// as bytes, codes 0-3 in .x.
__device__ __noinline__ uint2 quant8_exact(uint4 xv, const float4* tab, int stride, float qm) {
  const __half2* h = reinterpret_cast<const __half2*>(&xv);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float x = (k & 1) ? __high2float(h[k >> 1]) : __low2float(h[k >> 1]);
    float4 sc = tab[k * stride];
    if (qm >= 0.0f) sc.w = qm;
    const uint32_t q = quant_fast(x, sc);
    if (k < 4) lo |= q << (8 * k);
    else hi |= q << (8 * (k - 4));
  }
  return make_uint2(lo, hi);
}

// Two fp32 lanes in one 64-bit register: paired IEEE operations, each lane
// rounded exactly like the scalar instruction.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2unpack(uint64_t d, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Eight codes of one 16-byte chunk, branch-free on the common path, two
// elements per paired operation: 0 <= y < 2^22, so y + 2^23 rounds y to the
// nearest integer (ties to even) and that integer sits in the low mantissa
// bits.  A chunk with any quotient near a rounding boundary is redone element
// by element by quant8_exact.  mn2[j], r2[j]: (min, 1/s) of elements 2j,
// 2j+1; qmax is the same for all eight; tab/stride/qm: the scales in shared
// memory for the exact path.
__device__ __forceinline__ void quant8(const uint4& xv, const uint64_t (&mn2)[4], const uint64_t (&r2)[4],
                                       uint32_t qmax, const float4* tab, int stride, float qm,
                                       uint32_t (&code)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&xv);
  const uint64_t magic = f2pack(8388608.0f, 8388608.0f);
  bool near = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 xf = __half22float2(h[j]);
    const uint64_t y = f2mul(f2sub(f2pack(xf.x, xf.y), mn2[j]), r2[j]);
    const uint64_t t = f2add(y, magic);
    float d0, d1, t0, t1;
    f2unpack(f2sub(y, f2sub(t, magic)), d0, d1);
    near |= (fabsf(d0) >= kNearHalf) | (fabsf(d1) >= kNearHalf);
    f2unpack(t, t0, t1);
    const uint32_t c0 = __float_as_uint(t0) - 0x4B000000u, c1 = __float_as_uint(t1) - 0x4B000000u;
    code[2 * j] = c0 < qmax ? c0 : qmax;
    code[2 * j + 1] = c1 < qmax ? c1 : qmax;
  }
  if (near) {
    const uint2 b = quant8_exact(xv, tab, stride, qm);
#pragma unroll
    for (int k = 0; k < 8; ++k) code[k] = ((k < 4 ? b.x : b.y) >> (8 * (k & 3))) & 0xFFu;
  }
}

// Quantizes one staged group (rows of the stage are the group's G tokens; a
// row that came from the ring has its 16-byte chunks swizzled by t & 7) into
// the record staging area.  Thread (chunk c, row group rg) owns chunk c of
// rows rg + k*RG, k < RT, and keeps them in registers from the min/max pass
// to the code pass.  after_load() runs once every thread holds its rows (the
// stage may then be refilled: with 2- to 8-bit codes nothing reads it again).
template <int KB, int VB, int D, bool kWide, typename AfterLoad>
__device__ bool flush_group(const AppendParams& p, const __half* kt, const __half* vt, int nring, uint8_t* smem,
                            const AppendSmem& L, bool staged, AfterLoad&& after_load) {
  constexpr int WK = words_per_row(D, KB);
  constexpr int WV = words_per_row(D, VB);
  constexpr int CH = D / 8;     // 16-byte chunks per row
  constexpr int RT = kWide ? D / 16 : D / 32;  // rows per thread
  constexpr int LPC = 32 / CH;  // lanes of a warp on the same chunk
  const int G = p.G;
  const int RG = (kWide ? 2 : 4) * G / CH;     // row groups
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid % CH, rg = tid / CH;
  uint8_t* rec = smem + L.off_rec;
  uint32_t* kc = reinterpret_cast<uint32_t*>(rec);
  uint32_t* vc = kc + G * WK;
  // per-token keys (uniform for the launch): one (scale, zero) pair per token
  // instead of the per-channel scale and zero rows
  const bool ktok = p.key_mode == 1;
  __half* ks16 = reinterpret_cast<__half*>(vc + G * WV);
  __half* kz16 = ks16 + D;
  __half2* ksz = reinterpret_cast<__half2*>(vc + G * WV);
  __half2* vsz = ktok ? ksz + G : reinterpret_cast<__half2*>(kz16 + D);
  __half2* kpt = reinterpret_cast<__half2*>(smem + L.off_kpt);
  float4* ksct = reinterpret_cast<float4*>(smem + L.off_ksct);
  float4* ksc = reinterpret_cast<float4*>(smem + L.off_ksc);
  float4* vsc = reinterpret_cast<float4*>(smem + L.off_vsc);
  float* vr2 = reinterpret_cast<float*>(smem + L.off_vr2);
  __half* kmn = reinterpret_cast<__half*>(smem + L.off_kmn);
  __half* kmx = reinterpret_cast<__half*>(smem + L.off_kmx);
  __half2* vpart = reinterpret_cast<__half2*>(smem + L.off_vpart);
  auto key_of = [&](int t) { return t < nring ? (t & 7) : 0; };
  // channel scales are stored element-major ([k][chunk]) so that the lanes of
  // a row, one chunk each, read consecutive entries
  auto ksc_at = [&](int ch) -> float4& { return ksc[(ch & 7) * CH + (ch >> 3)]; };
  const uint4* kq = reinterpret_cast<const uint4*>(kt);
  const uint4* vq = reinterpret_cast<const uint4*>(vt);

  // ---- phase 1: load the thread's chunks; key min/max per channel (over
  // the thread's rows, then the warp's lanes on the chunk, then per warp in
  // shared memory); value min/max per token (the row's CH lanes)
  uint4 xk[RT], xv[RT];
#pragma unroll
  for (int k = 0; k < RT; ++k) {
    const int t = rg + k * RG;
    const int pc = c ^ key_of(t);
    xk[k] = kq[t * CH + pc];
    xv[k] = vq[t * CH + pc];
  }
  // (min, -max) of a row's chunks over its CH lanes: one min-reduction serves both
  auto row_minmax = [&](const uint4& x) -> __half2 {
    const __half2* h = reinterpret_cast<const __half2*>(&x);
    const __half2 m2 = __hmin2(__hmin2(h[0], h[1]), __hmin2(h[2], h[3]));
    const __half2 M2 = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    __half2 r = __halves2half2(__hmin(__low2half(m2), __high2half(m2)),
                               __hneg(__hmax(__low2half(M2), __high2half(M2))));
#pragma unroll
    for (int off = 1; off < CH; off <<= 1)
      r = __hmin2(r, u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(r), off)));
    return r;
  };
  if (ktok) {
#pragma unroll
    for (int k = 0; k < RT; ++k) {
      const __half2 r = row_minmax(xk[k]);
      if (c == 0) kpt[rg + k * RG] = r;
    }
  } else {
    __half2 mn[4], mx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mn[i] = reinterpret_cast<const __half2*>(&xk[0])[i];
      mx[i] = mn[i];
    }
#pragma unroll
    for (int k = 1; k < RT; ++k)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 x = reinterpret_cast<const __half2*>(&xk[k])[i];
        mn[i] = __hmin2(mn[i], x);
        mx[i] = __hmax2(mx[i], x);
      }
#pragma unroll
    for (int off = CH; off < 32; off <<= 1)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mn[i] = __hmin2(mn[i], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mn[i]), off)));
        mx[i] = __hmax2(mx[i], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mx[i]), off)));
      }
    if (lane < CH) {
      *reinterpret_cast<uint4*>(kmn + warp * D + 8 * c) =
          make_uint4(h2_as_u32(mn[0]), h2_as_u32(mn[1]), h2_as_u32(mn[2]), h2_as_u32(mn[3]));
      *reinterpret_cast<uint4*>(kmx + warp * D + 8 * c) =
          make_uint4(h2_as_u32(mx[0]), h2_as_u32(mx[1]), h2_as_u32(mx[2]), h2_as_u32(mx[3]));
    }
  }
#pragma unroll
  for (int k = 0; k < RT; ++k) {
    const __half2 r = row_minmax(xv[k]);
    if (c == 0) vpart[rg + k * RG] = r;
  }
  if (tid == 0) bulk_wait_read_all();  // the previous record has left the staging area
  // every thread saw its stage arrive, or all of them stop here
  if (__syncthreads_or(!staged)) return false;
  after_load();

  // ---- phase 2: one scale per thread (channel tid, token tid; per-token
  // keys: token tid - G)
  if (ktok) {
    if (KB != 3 && tid >= G && tid < 2 * G) {
      const int t = tid - G;
      const __half2 r = kpt[t];
      const Scale sc = make_scale<KB>(__low2half(r), __hneg(__high2half(r)), false);
      ksct[t] = make_float4(sc.mn, sc.s, sc.r, sc.qmax);
      ksz[t] = __halves2half2(sc.s16, sc.z16);
    }
  } else if (tid < D) {
    // thread tid takes channel 8*(tid % CH) + tid / CH, whose table slot is tid
    const int ch = 8 * (tid % CH) + tid / CH;
    const int warps = (kWide ? 2 : 4) * G / 32;
    __half mn = kmn[ch], mx = kmx[ch];
    for (int w = 1; w < warps; ++w) {
      mn = __hmin(mn, kmn[w * D + ch]);
      mx = __hmax(mx, kmx[w * D + ch]);
    }
    const Scale sc = make_scale<KB>(mn, mx, KB == 3 && ch % 11 == 10);
    ksc[tid] = make_float4(sc.mn, sc.s, sc.r, sc.qmax);
    {
      float* kpf = reinterpret_cast<float*>(smem + L.off_kp);
      const int pi = (((ch & 7) >> 1) * CH + (ch >> 3)) * 2 + (ch & 1);
      kpf[pi] = sc.mn;
      kpf[D + pi] = sc.r;
    }
    const int pos = KB == 3 ? ch : kscale_pos(ch, D);
    ks16[pos] = sc.s16;
    kz16[pos] = sc.z16;
  }
  // value scales: token vtk (wide CTAs with G >= D: the threads after the D
  // channel ones)
  const int vtk = (kWide && !ktok && G >= D) ? tid - D : tid;
  if (vtk >= 0 && vtk < G) {
    const __half2 r = vpart[vtk];
    const __half mn = __low2half(r), mx = __hneg(__high2half(r));
    const Scale s3 = make_scale<VB>(mn, mx, false);
    float s2 = s3.s, r2 = s3.r;
    if (VB == 3) {
      const Scale t2 = make_scale<VB>(mn, mx, true);
      s2 = t2.s;
      r2 = t2.r;
    }
    vsc[vtk] = make_float4(s3.mn, s3.s, s3.r, s2);
    vr2[vtk] = r2;
    vsz[vtk] = __halves2half2(s3.s16, s3.z16);
  }
  __syncthreads();

  // ---- phase 3: codes, packed LSB first into the record staging area
  // (the packing of a row's codes is the same for both key modes)
  auto put_k = [&](int t, const uint32_t (&code)[8]) {
    uint32_t w0, w1;
    pack8<KB>(code, w0, w1);
    const int xk = code_word_xor(WK, true, t);
    if (KB == 8) {
      *reinterpret_cast<uint2*>(kc + t * WK + ((2 * c) ^ xk)) = make_uint2(w0, w1);
    } else if (KB == 4) {
      kc[t * WK + (c ^ xk)] = w0;
    } else {  // KB == 2: two lanes form one word
      const uint32_t other = __shfl_xor_sync(0xffffffffu, w0, 1);
      if ((c & 1) == 0) kc[t * WK + ((c / 2) ^ xk)] = w0 | (other << 16);
    }
  };
  if (ktok) {
    if constexpr (KB != 3) {
#pragma unroll
      for (int k = 0; k < RT; ++k) {
        const int t = rg + k * RG;
        const float4 s = ksct[t];
        const uint64_t m = f2pack(s.x, s.x), r = f2pack(s.z, s.z);
        const uint64_t mn2[4] = {m, m, m, m}, r2[4] = {r, r, r, r};
        uint32_t code[8];
        quant8(xk[k], mn2, r2, (1u << KB) - 1, ksct + t, 0, -1.0f, code);
        put_k(t, code);
      }
    }
  } else if constexpr (KB != 3) {
    const uint64_t* kp = reinterpret_cast<const uint64_t*>(smem + L.off_kp);
    uint64_t mn2[4], r2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mn2[j] = kp[j * CH + c];
      r2[j] = kp[D / 2 + j * CH + c];
    }
#pragma unroll
    for (int k = 0; k < RT; ++k) {
      const int t = rg + k * RG;
      uint32_t code[8];
      quant8(xk[k], mn2, r2, (1u << KB) - 1, ksc + c, CH, -1.0f, code);
      put_k(t, code);
    }
  } else {
    for (int idx = tid; idx < G * WK; idx += blockDim.x) {
      const int t = idx / WK, w = idx - (idx / WK) * WK;
      const int key = key_of(t);
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 11; ++j) {
        const int ch = 11 * w + j;
        if (ch < D) {
          const __half x = kt[t * D + ((((ch >> 3) ^ key) << 3) | (ch & 7))];
          word |= quant_fast(__half2float(x), ksc_at(ch)) << (j == 10 ? 30 : 3 * j);
        }
      }
      kc[idx] = word;
    }
  }
  if constexpr (VB != 3) {
#pragma unroll
    for (int k = 0; k < RT; ++k) {
      const int t = rg + k * RG;
      const float4 s = vsc[t];
      const uint64_t m = f2pack(s.x, s.x), r = f2pack(s.z, s.z);
      const uint64_t mn2[4] = {m, m, m, m}, r2[4] = {r, r, r, r};
      uint32_t code[8];
      quant8(xv[k], mn2, r2, (1u << VB) - 1, vsc + t, 0, static_cast<float>((1 << VB) - 1), code);
      uint32_t w0, w1;
      pack8<VB>(code, w0, w1);
      const int xv = code_word_xor(WV, false, t);
      if (VB == 8) {
        *reinterpret_cast<uint2*>(vc + t * WV + ((2 * c) ^ xv)) = make_uint2(w0, w1);
      } else if (VB == 4) {
        vc[t * WV + (c ^ xv)] = w0;
      } else {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, w0, 1);
        if ((c & 1) == 0) vc[t * WV + ((c / 2) ^ xv)] = w0 | (other << 16);
      }
    }
  } else {
    for (int idx = tid; idx < G * WV; idx += blockDim.x) {
      const int t = idx / WV, w = idx - (idx / WV) * WV;
      const int key = key_of(t);
      const float4 s = vsc[t];
      const float4 s3 = make_float4(s.x, s.y, s.z, 7.0f);
      const float4 s2 = make_float4(s.x, s.w, vr2[t], 3.0f);
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 11; ++j) {
        const int ch = 11 * w + j;
        if (ch < D) {
          const __half x = vt[t * D + ((((ch >> 3) ^ key) << 3) | (ch & 7))];
          word |= quant_fast(__half2float(x), j == 10 ? s2 : s3) << (j == 10 ? 30 : 3 * j);
        }
      }
      vc[idx] = word;
    }
  }
  return true;
}

// Copy new tokens [lo, hi) (absolute positions, all from this call's input)
// into the unit's FP16 rings, 16-byte chunks swizzled by slot.  A thread
// issues up to four loads before its stores.
template <int D>
__device__ void write_residual(const AppendParams& p, int u, int64_t lo, int64_t hi, int64_t T) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const int n = static_cast<int>(hi - lo);
  const int base = static_cast<int>(lo - T);
  const int total = n * 2 * CH;
  const int step = blockDim.x;
  for (int idx0 = threadIdx.x; idx0 < total; idx0 += 4 * step) {
    uint4 v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int idx = idx0 + r * step;
      if (idx < total) {
        const int tok = idx / (2 * CH);
        const int rem = idx - tok * (2 * CH);
        const __half* in = rem >= CH ? p.V : p.K;
        v[r] = __ldg(reinterpret_cast<const uint4*>(in + (static_cast<int64_t>(u) * p.n + base + tok) * D) +
                     (rem % CH));
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int idx = idx0 + r * step;
      if (idx < total) {
        const int tok = idx / (2 * CH);
        const int rem = idx - tok * (2 * CH);
        __half* ring = rem >= CH ? p.res_v : p.res_k;
        const int slot = static_cast<int>((lo + tok) % p.R);
        uint4* dst = reinterpret_cast<uint4*>(ring + u * p.res_stride + static_cast<int64_t>(slot) * D) +
                     ((rem % CH) ^ (slot & 7));
        if (in_range(dst, 16, p.buf_lo, p.buf_hi, p.err)) *dst = v[r];  // (checked in debug builds)
      }
    }
  }
}

// Register budget of the 128-thread launches (G = 32 flushes, single-token
// appends, window writes): five CTAs per SM where five fit in shared memory
// (records without 8-bit codes), so that more independent CTAs cover each
// other's barrier waits; larger CTAs (G = 64, 128) take the 512-thread bound.
template <int KB, int VB>
__host__ __device__ constexpr int append_min_ctas_128() { return (KB == 8 || VB == 8) ? 4 : 5; }

template <int KB, int VB, int D, int TPB, int MINB, bool kWide>
__global__ void __launch_bounds__(TPB, MINB) append_kernel(AppendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const bool per_unit = (p.mode & kPerUnit) != 0;
  // single-token append: the token's K/V row is loaded while the counter is in flight
  constexpr int CH = D / 8;
  uint4 newrow = make_uint4(0u, 0u, 0u, 0u);
  if (per_unit && tid < 2 * CH) {
    const __half* in = tid >= CH ? p.V : p.K;
    newrow = __ldg(reinterpret_cast<const uint4*>(in + static_cast<int64_t>(blockIdx.x) * D) + (tid % CH));
  }
  // The window state.  A single-token append (one CTA per unit) reads its
  // unit's (tokens, quantized, bound) once per CTA, so that every thread works
  // from the same values even if a misordered launch changes them meanwhile,
  // and steps it (a decode step may shrink the bound and quantize several
  // groups).  A multi-token append takes the host's state.
  __shared__ int st_shared[4];
  if (tid == 0) {
    if (per_unit) {
      const int u = blockIdx.x;
      const int t = __ldcg(p.tokens + u);
      WindowState w0;
      w0.nq = __ldcg(p.nq + u);
      w0.bound = __ldcg(p.bound + u);
      const WindowState w1 = window_after_append(t, w0, 1, p.G, p.rpc);
      st_shared[0] = t;
      st_shared[1] = static_cast<int>(w0.nq);
      st_shared[2] = static_cast<int>(w1.nq);
      st_shared[3] = w1.bound;
    } else {
      st_shared[0] = p.T0;
      st_shared[1] = p.nq0;
      st_shared[2] = p.nq1;
      st_shared[3] = 0;
    }
  }
  __syncthreads();
  const int T = st_shared[0];
  const int nq0 = st_shared[1];
  const int nq1 = st_shared[2];

  if (p.mode & kFlush) {
    // jobs: a single-token append's CTA quantizes its unit's groups nq0/G ..
    // nq1/G - 1 in order; a multi-token append's job j is (unit j / nflush,
    // group nq0/G + j % nflush), CTA-strided.  job(k) is this CTA's k-th job.
    const AppendSmem L = append_smem_layout(D, p.G, p.rec_bytes, kWide);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bars);
    const int nflush = (nq1 - nq0) / p.G;
    const int njobs = per_unit ? nflush : nflush * p.units;
    const uint32_t tile = static_cast<uint32_t>(L.tile);
    auto job_valid = [&](int k) {
      return per_unit ? k < njobs : static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x) < njobs;
    };
    auto job_of = [&](int k, int& u, int& grp) {
      if (per_unit) {
        u = blockIdx.x;
        grp = nq0 / p.G + k;
      } else {
        const int j = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        u = j / nflush;
        grp = nq0 / p.G + (j - u * nflush);
      }
    };
    // stage the K and V rows of job k: ring rows first (slots of a group are
    // contiguous: the group starts at a multiple of G and R is one too), then
    // rows of this call's input
    auto issue = [&](int k, int st) {
      int u, grp;
      job_of(k, u, grp);
      const int t0 = grp * p.G;
      const int nring = T > t0 ? (T - t0 < p.G ? T - t0 : p.G) : 0;
      uint8_t* ks = smem + st * L.off_stage1;
      uint8_t* vs = ks + tile;
      if (nring > 0) {
        // (debug builds: ring rows outside the cache buffer are recorded; the
        // stage's barrier completes without copies)
        const int64_t r0 = u * p.res_stride + static_cast<int64_t>(t0 % p.R) * D;
        const size_t rb = static_cast<size_t>(nring) * D * 2;
        if (!in_range(p.res_k + r0, rb, p.buf_lo, p.buf_hi, p.err) || !in_range(p.res_v + r0, rb, p.buf_lo, p.buf_hi, p.err)) {
          mbar_arrive(&bars[st]);
          return;
        }
      }
      mbar_arrive_expect_tx(&bars[st], 2 * tile);
      if (nring > 0) {
        const int s0 = t0 % p.R;
        const uint32_t b = static_cast<uint32_t>(nring) * D * 2;
        bulk_g2s(ks, p.res_k + u * p.res_stride + static_cast<int64_t>(s0) * D, b, &bars[st]);
        bulk_g2s(vs, p.res_v + u * p.res_stride + static_cast<int64_t>(s0) * D, b, &bars[st]);
      }
      if (nring < p.G) {
        const int64_t row = static_cast<int64_t>(u) * p.n + (t0 + nring - T);
        const uint32_t b = static_cast<uint32_t>(p.G - nring) * D * 2;
        const uint32_t o = static_cast<uint32_t>(nring) * D * 2;
        bulk_g2s(ks + o, p.K + row * D, b, &bars[st]);
        bulk_g2s(vs + o, p.V + row * D, b, &bars[st]);
      }
    };
    if (tid == 0) {
      mbar_init(&bars[0], 1);
      mbar_init(&bars[1], 1);
      fence_mbar_init();
      if (job_valid(0)) issue(0, 0);
      if (!kWide && job_valid(1)) issue(1, 1);
    }
    __syncthreads();
    for (int k = 0; job_valid(k); ++k) {
      // two stages alternate; a wide CTA's single stage completes once per job
      const int st = kWide ? 0 : (k & 1);
      const uint32_t parity = static_cast<uint32_t>(kWide ? (k & 1) : ((k >> 1) & 1));
      int u, grp;
      job_of(k, u, grp);
      const int t0 = grp * p.G;
      const int nring = T > t0 ? (T - t0 < p.G ? T - t0 : p.G) : 0;
      const bool ok = mbar_wait(&bars[st], parity, p.err);
      const __half* kt = reinterpret_cast<const __half*>(smem + st * L.off_stage1);
      auto refill = [&]() {
        if (kWide && tid == 0 && job_valid(k + 1)) issue(k + 1, 0);
      };
      if (!flush_group<KB, VB, D, kWide>(p, kt, kt + p.G * D, nring, smem, L, ok, refill)) {
        // a copy never landed (all threads agree): give the other stage's copy
        // its bounded wait, then stop (a wide CTA has issued no other copy)
        if (!kWide && job_valid(k + 1)) mbar_wait(&bars[st ^ 1], static_cast<uint32_t>(((k + 1) >> 1) & 1), p.err);
        break;
      }
      __syncthreads();  // stage and record staging complete
      if (tid == 0) {
        fence_proxy_async_smem();
        uint8_t* dst = p.records + static_cast<int64_t>(u) * p.unit_rec_stride + static_cast<int64_t>(grp) * p.rec_bytes;
        if (in_range(dst, static_cast<size_t>(p.rec_bytes), p.buf_lo, p.buf_hi, p.err))  // debug builds
          bulk_s2g(dst, smem + L.off_rec, static_cast<uint32_t>(p.rec_bytes));
        bulk_commit();
        if (!kWide && job_valid(k + 2)) issue(k + 2, st);
      }
    }
    if (tid == 0) bulk_wait_all();
  }
  if (p.mode & kResidual) {
    // tokens that stay in the window after this call
    const int first = T > nq1 ? T : nq1;
    const int last = T + p.n;
    if (per_unit) {  // single token: CTA u writes unit u's token unless it was flushed
      if (first < last && tid < 2 * CH) {
        __half* ring = tid >= CH ? p.res_v : p.res_k;
        const int slot = T % p.R;
        reinterpret_cast<uint4*>(ring + blockIdx.x * p.res_stride + static_cast<int64_t>(slot) * D)[(tid % CH) ^ (slot & 7)] =
            newrow;
      }
    } else {
      const int lo = first + static_cast<int>(blockIdx.x) * 16;
      const int hi = (lo + 16 < last) ? lo + 16 : last;
      if (lo < hi) write_residual<D>(p, blockIdx.y, lo, hi, T);
    }
  }
  if (p.mode & kUpdateState) {
    if (per_unit) {
      // the next kernel on the stream sees it; no CTA of this launch reads it again
      if (tid == 0) {
        p.tokens[blockIdx.x] = T + p.n;
        p.nq[blockIdx.x] = nq1;
        p.bound[blockIdx.x] = st_shared[3];
      }
    } else {
      // the last CTA to finish advances every unit's counter
      __shared__ int last;
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        last = atomicAdd(p.done_ctr, 1) == p.ctas - 1;
      }
      __syncthreads();
      if (last) {  // (a multi-token append keeps the bound)
        for (int u = tid; u < p.units; u += blockDim.x) {
          p.tokens[u] = T + p.n;
          p.nq[u] = nq1;
        }
        if (tid == 0) *p.done_ctr = 0;
      }
    }
  }
}

}  // namespace

// The instantiation for a launch of `threads` threads: wide G = 128 flushes
// (256 threads, two CTAs per SM), 128-thread flushes (G = 32) and window
// writes, or the 512-thread bound for the other G = 64 and 128 flushes.
template <int KB, int VB, int D>
static void (*append_kernel_for(int threads, int G))(AppendParams) {
  if constexpr (append_wide(KB, VB, 128)) {
    if (G == 128 && threads == append_threads(128, true)) return append_kernel<KB, VB, D, 256, 2, true>;
  }
  if (threads <= 128) return append_kernel<KB, VB, D, 128, append_min_ctas_128<KB, VB>(), false>;
  return append_kernel<KB, VB, D, 512, 1, false>;
}

template <int KB, int VB, int D>
static cudaError_t launch_append(const AppendParams& p, dim3 grid, int threads, size_t smem, cudaStream_t s) {
  auto k = append_kernel_for<KB, VB, D>(threads, p.G);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  k<<<grid, threads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int KB, int VB, int D>
static int occupancy_append(int threads, int G, size_t smem) {
  auto k = append_kernel_for<KB, VB, D>(threads, G);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, threads, smem) != cudaSuccess) return 0;
  return occ;
}

#define KVQ_APPEND_ENTRY(KB, VB)                                                     \
  case (KB * 16 + VB):                                                              \
    return D == 128 ? launch_append<KB, VB, 128>(p, grid, threads, smem, s)         \
                    : launch_append<KB, VB, 64>(p, grid, threads, smem, s);

cudaError_t append_dispatch(int kb, int vb, int D, const AppendParams& p, dim3 grid, int threads, size_t smem,
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
#undef KVQ_APPEND_ENTRY

#define KVQ_APPEND_OCC(KB, VB) \
  case (KB * 16 + VB):        \
    return D == 128 ? occupancy_append<KB, VB, 128>(threads, G, smem) : occupancy_append<KB, VB, 64>(threads, G, smem);

int append_ctas_per_sm(int kb, int vb, int D, int G, int threads, size_t smem) {
  switch (kb * 16 + vb) {
    KVQ_APPEND_OCC(2, 2) KVQ_APPEND_OCC(2, 3) KVQ_APPEND_OCC(2, 4) KVQ_APPEND_OCC(2, 8)
    KVQ_APPEND_OCC(3, 2) KVQ_APPEND_OCC(3, 3) KVQ_APPEND_OCC(3, 4) KVQ_APPEND_OCC(3, 8)
    KVQ_APPEND_OCC(4, 2) KVQ_APPEND_OCC(4, 3) KVQ_APPEND_OCC(4, 4) KVQ_APPEND_OCC(4, 8)
    KVQ_APPEND_OCC(8, 2) KVQ_APPEND_OCC(8, 3) KVQ_APPEND_OCC(8, 4) KVQ_APPEND_OCC(8, 8)
    default:
      return 0;
  }
}
#undef KVQ_APPEND_OCC

int append_block_threads(int kb, int vb, int G) { return append_threads(G, append_wide(kb, vb, G)); }

size_t append_smem_bytes(int kb, int vb, int D, int G, int rec_bytes) {
  return static_cast<size_t>(append_smem_layout(D, G, rec_bytes, append_wide(kb, vb, G)).total);
}

}  // namespace kvq
