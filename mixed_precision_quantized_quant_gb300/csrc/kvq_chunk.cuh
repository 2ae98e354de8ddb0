// Causal multi-query attention over one layer's quantized cache: the queries
// of the n newest tokens attend every cached token at or before their own
// position, quantized groups dequantized and window tokens exact.  KVTuner
// (section A2, calibration design) runs prefill attention this way, over the
// dequantized cache; the attention itself is its A3 equation.
//
// One CTA of 256 threads owns 256 (query, head) rows of one (batch, kv head)
// unit, as two groups of 128 rows (one MMA tile each, one thread per row),
// and walks the unit's tokens in tiles of 64, first the quantized groups and
// then the FP16 window.  Per tile:
//   1. all threads unpack the tile into shared memory as MMA operands, once
//      for both groups:
//      keys k^ = code*s + z in fp32, split into fp16 hi + lo halves (so the
//      products keep about 22 bits); value codes as exact fp16 integers, the
//      window's values as they are; the per-token value (scale, zero).
//   2. one thread issues S = Q K^T as tcgen05 MMAs (hi and lo) into tensor
//      memory (128 lanes x 64 fp32 columns per group), group 0 first.
//   3. each thread loads its row of S from tensor memory and runs the online
//      softmax in the log2 domain (lazy rescale: only when the running max
//      grows by more than 2^8).  It writes P' = p * s_value as fp16 hi + lo
//      rows and keeps l = sum p and zs = sum p * z_value in registers, so the
//      value zero never enters an MMA.
//   4. one thread per group issues O += P' C (hi and lo) into tensor memory
//      (128 lanes x d fp32 columns per group), C being the value codes.
// Group 0's softmax runs while group 1's score MMAs do, and group 1's while
// group 0's P.V MMAs do.
// The epilogue returns (O + zs) / l.  3-bit value rows store their 2-bit
// field (channel 11w + 10) with scale s2 = (7 s)/3; those codes enter C as
// 7 * code, and their O columns are divided by 3 once before the window
// tiles (or in the epilogue when there are none).
//
// Operands in shared memory use the no-swizzle core-matrix layout: Q, K^ hi,
// K^ lo and P' are K-major; the values are stored token-major, which is the
// MN-major form of the P.V product's B operand.
#pragma once

#include <cuda_fp16.h>

#include "kvq_kernels.h"
#include "kvq_tc.cuh"

namespace kvq {

constexpr int kChunkRows = 256;     // (query, head) rows per CTA: two groups
constexpr int kChunkM = 128;        // rows per group: the MMA's M
constexpr int kChunkTile = 64;      // tokens per tile: N of the score MMA, K of P.V
constexpr int kChunkThreads = 256;  // one thread per row

template <int D>
struct ChunkSmem {
  static constexpr int KC = D / 8;                                  // core matrices along d
  static constexpr uint32_t q = 0;                                  // [256 rows][D] f16
  static constexpr uint32_t kh = q + kChunkRows * D * 2;            // [64 tokens][D] f16, hi
  static constexpr uint32_t kl = kh + kChunkTile * D * 2;           // lo
  static constexpr uint32_t ph = kl + kChunkTile * D * 2;           // [256 rows][64 tokens] f16, hi
  static constexpr uint32_t pl = ph + kChunkRows * kChunkTile * 2;  // lo
  static constexpr uint32_t pgroup = kChunkM * kChunkTile * 2;      // bytes of one group's P
  static constexpr uint32_t v = pl + kChunkRows * kChunkTile * 2;   // [64 tokens][D] f16
  static constexpr uint32_t ts = v + D * kChunkTile * 2;            // value scale per token, f32
  static constexpr uint32_t tz = ts + kChunkTile * 4;               // value zero per token, f32
  static constexpr uint32_t bars = tz + kChunkTile * 4;             // mbarriers: S[2], O[2]
  static constexpr uint32_t tslot = bars + 32;                      // tensor-memory address
  static constexpr uint32_t bytes = tslot + 16;
  // tensor memory: S of group g in columns [64 g, 64 g + 64), O of group g
  // in [128 + D g, 128 + D g + D)
  static constexpr uint32_t tcols = D == 128 ? 512 : 256;
};

// Unpacking plan of one thread's 8 channels c0 .. c0+7 of a B-bit code row
// (fields least significant first; 3-bit words hold ten 3-bit fields and a
// 2-bit one in bits 30..31).  Built once per thread.
template <int B>
struct Unpack8 {
  int wa = 0;         // word holding channel c0
  uint32_t sh0 = 0;   // B in {2, 4, 8}: bit offset of channel c0 in word wa
  uint64_t sh8 = 0;   // B = 3: byte e = shift of channel c0 + e
  uint32_t sel = 0;   // B = 3: bit e set if channel c0 + e is in word wa + 1
  uint32_t two = 0;   // B = 3: bit e set if channel c0 + e is the 2-bit field
  __device__ __forceinline__ void init(int c0) {
    if constexpr (B == 3) {
      wa = c0 / 11;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = c0 + e, w = c / 11, f = c - 11 * w;
        sh8 |= static_cast<uint64_t>(3 * f) << (8 * e);
        if (w != wa) sel |= 1u << e;
        if (f == 10) two |= 1u << e;
      }
    } else {
      wa = (c0 * B) >> 5;
      sh0 = static_cast<uint32_t>((c0 * B) & 31);
    }
  }
  __device__ __forceinline__ bool second_word() const { return B == 8 || (B == 3 && sel != 0u); }
  // code of channel c0 + e (e a constant after unrolling); w0 pre-shifted by sh0
  __device__ __forceinline__ uint32_t get(uint32_t w0, uint32_t w1, int e) const {
    if constexpr (B == 3) {
      const uint32_t w = ((sel >> e) & 1u) ? w1 : w0;
      const uint32_t s = static_cast<uint32_t>(sh8 >> (8 * e)) & 31u;
      return (w >> s) & (((two >> e) & 1u) ? 3u : 7u);
    } else if constexpr (B == 8) {
      return ((e < 4 ? w0 : w1) >> (8 * (e & 3))) & 0xFFu;
    } else {
      return (w0 >> (B * e)) & ((1u << B) - 1u);
    }
  }
};

__device__ __forceinline__ uint32_t pack_h2(__half a, __half b) {
  return static_cast<uint32_t>(__half_as_ushort(a)) | (static_cast<uint32_t>(__half_as_ushort(b)) << 16);
}

// two fp32 values as fp16 hi and lo halves: x ~ hi + lo to about 22 bits
__device__ __forceinline__ void split_hi_lo(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = h2_as_u32(h);
  lo = h2_as_u32(__floats2half2_rn(a - hf.x, b - hf.y));
}

// barrier of the 128 threads of one row group (ids 1 and 2; 0 is the CTA's)
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// exact small integer code (< 1024) as fp32: 2^23 + code, minus 2^23
__device__ __forceinline__ float code_f32(uint32_t c) { return __uint_as_float(0x4B000000u | c) - 8388608.0f; }

template <int KB, int VB, int D>
__global__ void __launch_bounds__(kChunkThreads, 1) chunk_attn_kernel(ChunkParams p) {
  using L = ChunkSmem<D>;
  constexpr int KC = L::KC;
  constexpr int kTile = kChunkTile;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* barS = reinterpret_cast<uint64_t*>(sm + L::bars);  // [2]: S of group g ready
  uint64_t* barO = barS + 2;                                   // [2]: P.V of group g done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::tslot);
  float* tok_s = reinterpret_cast<float*>(sm + L::ts);
  float* tok_z = reinterpret_cast<float*>(sm + L::tz);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int grp = tid >> 7;  // row group: rows 128 grp .. 128 grp + 127

  const int u = blockIdx.y;
  const int blk = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);  // longest rows first
  const int b = u / p.kv_heads, hk = u - b * p.kv_heads;
  const int i0 = blk * p.qpb;
  const int nqb = min(p.qpb, p.n - i0);
  const int rows = nqb * p.gqa;
  const int pos0 = p.T - p.n;  // position of query 0
  const int last_pos = pos0 + i0 + nqb - 1;
  const int gs = p.gshift;     // G = 1 << gs
  const uint8_t* urec = p.records + static_cast<int64_t>(u) * p.unit_rec_stride;
  const __half* rk = p.res_k + static_cast<int64_t>(u) * p.res_stride;
  const __half* rv = p.res_v + static_cast<int64_t>(u) * p.res_stride;

  // ---- query rows -> shared memory (row r = query r / gqa, head r % gqa)
  // (8 consecutive threads fill one 128-byte core matrix: conflict-free stores)
#pragma unroll 1
  for (int idx = tid; idx < kChunkRows * KC; idx += kChunkThreads) {
    const int r = (idx & 7) + 8 * (idx / (8 * KC)), kc = (idx >> 3) & (KC - 1);
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) {
      const int i = i0 + r / p.gqa, hh = r % p.gqa;
      const int64_t row = (static_cast<int64_t>(b) * p.Hq + hk * p.gqa + hh) * p.n + i;
      val = *reinterpret_cast<const uint4*>(p.q + row * D + kc * 8);
    }
    *reinterpret_cast<uint4*>(sm + L::q + core_off(r, kc * 8, KC)) = val;
  }
  if (tid == 0) {
    mbar_init(barS, 1);
    mbar_init(barS + 1, 1);
    mbar_init(barO, 1);
    mbar_init(barO + 1, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, L::tcols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = *tslot;
  const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  // this warp's lanes of its group's S and O
  const uint32_t tS = tb + kTile * grp + lane_off, tO = tb + 2 * kTile + D * grp + lane_off;
  const uint32_t sq = smem_u32(sm + L::q);
  const uint32_t skh = smem_u32(sm + L::kh), skl = smem_u32(sm + L::kl);
  const uint32_t sph = smem_u32(sm + L::ph), spl = smem_u32(sm + L::pl), sv = smem_u32(sm + L::v);
  constexpr uint32_t idS = idesc_f16_f32(kChunkM, kTile);
  constexpr uint32_t idO = idesc_f16_f32(kChunkM, D) | (1u << 16);  // B (values) MN-major

  // ---- fill coordinates.  Thread (tid & 7) fills row tid & 7 of every core
  // matrix it touches, so 8 consecutive threads store one whole 128-byte
  // core matrix; its channel octet kc is fixed and its tokens are
  // row0 + kStep * j.
  constexpr int kJ = kTile * KC / kChunkThreads;  // 16-byte chunks per thread per operand
  constexpr int kStep = kChunkThreads / KC;       // token stride between them
  const int kc = (tid >> 3) & (KC - 1);
  const int c0 = kc * 8;
  const int row0 = (tid & 7) + 8 * (tid / (8 * KC));
  Unpack8<KB> ku;
  Unpack8<VB> vu;
  ku.init(c0);
  vu.init(c0);
  const int voff = p.G * p.wk;  // value code rows follow the key code rows

  // ---- row state: this thread's row and the last position it may see
  const int r = tid;
  const int lim = (r < rows) ? pos0 + i0 + r / p.gqa : last_pos;
  float m = -INFINITY, l = 0.0f, zs = 0.0f;

  const int endQ = min(p.n_q, last_pos + 1);
  const int ntq = (endQ + kTile - 1) / kTile;
  const int endW = last_pos + 1;
  const int ntw = endW > p.n_q ? (endW - p.n_q + kTile - 1) / kTile : 0;
  const int ntiles = ntq + ntw;
  bool failed = false;

  // ---- words of one quantized tile, loaded a tile ahead of their use
  struct {
    uint32_t kw0[kJ], kw1[kJ], vw0[kJ], vw1[kJ];
    __half2 ksz[kJ];
    uint4 sa, za, sb, zb;  // per-channel key scales and zeros of groups gA, gB
    __half2 tsz;           // value (scale, zero) of token t0 + tid (tid < 64)
    int gA;
  } pf;
  auto prefetch = [&](int t0) {
    const int tq_end = min(t0 + kTile, p.n_q);  // whole groups: the rows exist
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int t = t0 + row0 + kStep * j;
      pf.kw0[j] = pf.kw1[j] = pf.vw0[j] = pf.vw1[j] = 0u;
      pf.ksz[j] = __floats2half2_rn(0.0f, 0.0f);
      if (t < tq_end) {
        const int gi = t >> gs, rr = t - (gi << gs);
        const uint8_t* rec = urec + static_cast<int64_t>(gi) * p.rec_bytes;
        const uint32_t* krow = reinterpret_cast<const uint32_t*>(rec) + rr * p.wk;
        const uint32_t* vrow = reinterpret_cast<const uint32_t*>(rec) + voff + rr * p.wv;
        pf.kw0[j] = krow[ku.wa];
        if (ku.second_word()) pf.kw1[j] = krow[ku.wa + 1];
        pf.vw0[j] = vrow[vu.wa];
        if (vu.second_word()) pf.vw1[j] = vrow[vu.wa + 1];
        if (p.km) pf.ksz[j] = *reinterpret_cast<const __half2*>(rec + p.off_kscale + rr * 4);
      }
    }
    // groups of the thread's first and last token, both below n_q / G
    pf.gA = min(t0 + row0, tq_end - 1) >> gs;
    const int gB = min(t0 + row0 + kStep * (kJ - 1), tq_end - 1) >> gs;
    if (p.km == 0) {
      const uint8_t* recA = urec + static_cast<int64_t>(pf.gA) * p.rec_bytes + p.off_kscale;
      const uint8_t* recB = urec + static_cast<int64_t>(gB) * p.rec_bytes + p.off_kscale;
      pf.sa = *reinterpret_cast<const uint4*>(recA + c0 * 2);
      pf.za = *reinterpret_cast<const uint4*>(recA + D * 2 + c0 * 2);
      pf.sb = *reinterpret_cast<const uint4*>(recB + c0 * 2);
      pf.zb = *reinterpret_cast<const uint4*>(recB + D * 2 + c0 * 2);
    }
    pf.tsz = __floats2half2_rn(0.0f, 0.0f);
    if (tid < kTile && t0 + tid < tq_end) {
      const int t = t0 + tid, gi = t >> gs, rr = t - (gi << gs);
      pf.tsz = *reinterpret_cast<const __half2*>(urec + static_cast<int64_t>(gi) * p.rec_bytes + p.off_vsz + rr * 4);
    }
  };
  if (ntq > 0) prefetch(0);

#pragma unroll 1
  for (int it = 0; it < ntiles; ++it) {
    const bool quant = it < ntq;
    const int t0 = quant ? it * kTile : p.n_q + (it - ntq) * kTile;
    const int tend = quant ? min(t0 + kTile, endQ) : min(t0 + kTile, endW);
    // the previous P.V product has read its operands (and written O)
    if (it > 0 && !failed) failed = !mbar_wait(barO, (it - 1) & 1, p.err) || !mbar_wait(barO + 1, (it - 1) & 1, p.err);

    // ---- keys (hi + lo halves) and values of the tile into shared memory,
    // from the words prefetched during the previous tile
    if (quant) {
      const int tq_end = min(t0 + kTile, p.n_q);
      float sA[8], zA[8], sB[8], zB[8];
      if (p.km == 0) {
        const __half* psa = reinterpret_cast<const __half*>(&pf.sa);
        const __half* pza = reinterpret_cast<const __half*>(&pf.za);
        const __half* psb = reinterpret_cast<const __half*>(&pf.sb);
        const __half* pzb = reinterpret_cast<const __half*>(&pf.zb);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sA[e] = __half2float(psa[e]);
          zA[e] = __half2float(pza[e]);
          sB[e] = __half2float(psb[e]);
          zB[e] = __half2float(pzb[e]);
          if constexpr (KB == 3) {
            if ((ku.two >> e) & 1u) {
              sA[e] = __fdiv_rn(__fmul_rn(sA[e], 7.0f), 3.0f);
              sB[e] = __fdiv_rn(__fmul_rn(sB[e], 7.0f), 3.0f);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int nn = row0 + kStep * j;
        const int t = t0 + nn;
        const bool inB = (t >> gs) != pf.gA;
        const uint32_t k0 = KB == 2 ? (pf.kw0[j] >> ku.sh0) : pf.kw0[j];
        const uint32_t v0 = VB == 2 ? (pf.vw0[j] >> vu.sh0) : pf.vw0[j];
        uint32_t hw[4], lw[4], vh[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          float kv[2];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            float s, z;
            if (p.km == 0) {
              s = inB ? sB[e + q2] : sA[e + q2];
              z = inB ? zB[e + q2] : zA[e + q2];
            } else {
              const float2 sz = __half22float2(pf.ksz[j]);
              s = sz.x;
              z = sz.y;
              if constexpr (KB == 3) {
                if ((ku.two >> (e + q2)) & 1u) s = __fdiv_rn(__fmul_rn(s, 7.0f), 3.0f);
              }
            }
            kv[q2] = fmaf(code_f32(ku.get(k0, pf.kw1[j], e + q2)), s, z);
          }
          split_hi_lo(kv[0], kv[1], hw[e / 2], lw[e / 2]);
          // value codes (< 1024) as exact fp16 integers: (1024 + code) - 1024
          uint32_t c_lo = vu.get(v0, pf.vw1[j], e), c_hi = vu.get(v0, pf.vw1[j], e + 1);
          if constexpr (VB == 3) {
            if ((vu.two >> e) & 1u) c_lo *= 7u;
            if ((vu.two >> (e + 1)) & 1u) c_hi *= 7u;
          }
          const uint32_t mag = 0x64006400u | c_lo | (c_hi << 16);
          vh[e / 2] = h2_as_u32(__hsub2(u32_as_h2(mag), __float2half2_rn(1024.0f)));
        }
        const bool live = t < tq_end;
        const uint32_t off = core_off(nn, c0, KC);
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sm + L::kh + off) = live ? make_uint4(hw[0], hw[1], hw[2], hw[3]) : zero;
        *reinterpret_cast<uint4*>(sm + L::kl + off) = live ? make_uint4(lw[0], lw[1], lw[2], lw[3]) : zero;
        *reinterpret_cast<uint4*>(sm + L::v + off) = live ? make_uint4(vh[0], vh[1], vh[2], vh[3]) : zero;
      }
      if (tid < kTile) {
        const bool vis = t0 + tid < tend;
        tok_s[tid] = vis ? __low2float(pf.tsz) : 0.0f;
        tok_z[tid] = vis ? __high2float(pf.tsz) : 0.0f;
      }
    } else {
      const int tw_end = min(t0 + kTile, p.T);
      uint4 kr[kJ], vr[kJ];
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int t = t0 + row0 + kStep * j;
        kr[j] = vr[j] = make_uint4(0u, 0u, 0u, 0u);
        if (t < tw_end) {
          const int slot = t % p.R;
          const int64_t off = static_cast<int64_t>(slot) * D + ((kc ^ (slot & 7)) * 8);
          kr[j] = *reinterpret_cast<const uint4*>(rk + off);
          vr[j] = *reinterpret_cast<const uint4*>(rv + off);
        }
      }
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const uint32_t off = core_off(row0 + kStep * j, c0, KC);
        *reinterpret_cast<uint4*>(sm + L::kh + off) = kr[j];
        *reinterpret_cast<uint4*>(sm + L::kl + off) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sm + L::v + off) = vr[j];
      }
    }
    if (!quant && tid < kTile) {
      tok_s[tid] = t0 + tid < tend ? 1.0f : 0.0f;
      tok_z[tid] = 0.0f;
    }
    // prefetch the next quantized tile's words; they land during this tile's MMAs and softmax
    if (it + 1 < ntq) prefetch((it + 1) * kTile);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    failed = __syncthreads_or(failed);

    // ---- S = Q K^T (hi, then lo), group 0 then group 1
    if (tid == 0 && !failed) {
      tc_fence_after_sync();
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint32_t qg = sq + g * (kChunkM * D * 2);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_f16(tb + kTile * g, smem_desc(qg + ks * 256, 128, KC * 128), smem_desc(skh + ks * 256, 128, KC * 128),
                   idS, ks > 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_f16(tb + kTile * g, smem_desc(qg + ks * 256, 128, KC * 128), smem_desc(skl + ks * 256, 128, KC * 128),
                   idS, 1u);
        umma_commit(barS + g);
      }
    }
    if (!failed) failed = !mbar_wait(barS + grp, it & 1, p.err);
    tc_fence_after_sync();

    // ---- online softmax of this thread's row
    float x[kTile];
#pragma unroll
    for (int c = 0; c < kTile; c += 16) {
      uint32_t rr[16];
      tmem_ld16(tS + c, rr);
      tmem_ld_wait(rr);
#pragma unroll
      for (int j = 0; j < 16; ++j) x[c + j] = __uint_as_float(rr[j]);
    }
    // tokens t0 .. t0 + nvis - 1 are visible to this row
    const int nvis = min(tend, lim + 1) - t0;
    float mx = -INFINITY;
    if (__all_sync(0xffffffffu, nvis >= kTile)) {
#pragma unroll
      for (int j = 0; j < kTile; ++j) mx = fmaxf(mx, x[j]);
    } else {
#pragma unroll
      for (int j = 0; j < kTile; ++j) {
        x[j] = j < nvis ? x[j] : -INFINITY;
        mx = fmaxf(mx, x[j]);
      }
    }
    // scores are raw q.k; the log2-domain max is m, in units of alpha * q.k
    mx *= p.alpha;
    const bool need = mx > m + 8.0f;
    float f = 1.0f;
    if (need) {
      f = ex2(m - mx);
      m = mx;
    }
    const float nm = -m;
    l *= f;
    zs *= f;
    // O *= f where the max moved; 3-bit values: divide the 2-bit-field
    // columns by 3 when the quantized tiles end
    const bool third = VB == 3 && it == ntq && ntq > 0;
    if (it > 0 && (__any_sync(0xffffffffu, need) || third)) {
#pragma unroll 1
      for (int c = 0; c < D; c += 16) {
        uint32_t o[16];
        tmem_ld16(tO + c, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float g = f;
          if (third && (c + j) % 11 == 10) g = __fdiv_rn(g, 3.0f);
          o[j] = __float_as_uint(__uint_as_float(o[j]) * g);
        }
        tmem_st16(tO + c, o);
      }
      tmem_st_wait();
    }
    float ls = 0.0f, zsum = 0.0f;
    uint32_t hi[kTile / 2], lo[kTile / 2];
#pragma unroll
    for (int j = 0; j < kTile; j += 2) {
      const float p0 = ex2(fmaf(x[j], p.alpha, nm)), p1 = ex2(fmaf(x[j + 1], p.alpha, nm));
      const float2 s2 = *reinterpret_cast<const float2*>(tok_s + j);
      const float2 z2 = *reinterpret_cast<const float2*>(tok_z + j);
      ls += p0 + p1;
      zsum = fmaf(p0, z2.x, fmaf(p1, z2.y, zsum));
      split_hi_lo(p0 * s2.x, p1 * s2.y, hi[j / 2], lo[j / 2]);
    }
    l += ls;
    zs += zsum;
#pragma unroll
    for (int cc = 0; cc < kTile / 8; ++cc) {
      *reinterpret_cast<uint4*>(sm + L::ph + grp * L::pgroup + core_off(r & 127, 8 * cc, kTile / 8)) =
          make_uint4(hi[4 * cc], hi[4 * cc + 1], hi[4 * cc + 2], hi[4 * cc + 3]);
      *reinterpret_cast<uint4*>(sm + L::pl + grp * L::pgroup + core_off(r & 127, 8 * cc, kTile / 8)) =
          make_uint4(lo[4 * cc], lo[4 * cc + 1], lo[4 * cc + 2], lo[4 * cc + 3]);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    group_sync(1 + grp);

    // ---- O += P' C (hi, then lo) of this group; C token-major (MN-major B)
    if ((tid & 127) == 0 && !failed) {
      tc_fence_after_sync();
      const uint32_t dO = tb + 2 * kTile + D * grp;
      const uint32_t pg = grp * L::pgroup;
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks)
        umma_f16(dO, smem_desc(sph + pg + ks * 256, 128, (kTile / 8) * 128),
                 smem_desc(sv + ks * 2 * KC * 128, KC * 128, 128), idO, (it > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks)
        umma_f16(dO, smem_desc(spl + pg + ks * 256, 128, (kTile / 8) * 128),
                 smem_desc(sv + ks * 2 * KC * 128, KC * 128, 128), idO, 1u);
      umma_commit(barO + grp);
    }
  }

  // ---- epilogue: out = (O + zs) / l
  if (!failed) failed = !mbar_wait(barO + grp, (ntiles - 1) & 1, p.err);
  tc_fence_after_sync();
  const bool third = VB == 3 && ntw == 0;
  const float inv = 1.0f / l;
  float* orow = nullptr;
  if (r < rows) {
    const int i = i0 + r / p.gqa, hh = r % p.gqa;
    orow = p.out + ((static_cast<int64_t>(b) * p.Hq + hk * p.gqa + hh) * p.n + i) * D;
  }
#pragma unroll 1
  for (int c = 0; c < D; c += 16) {
    uint32_t o[16];
    tmem_ld16(tO + c, o);
    tmem_ld_wait(o);
    if (orow) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float a = __uint_as_float(o[j]);
        if (third && (c + j) % 11 == 10) a = __fdiv_rn(a, 3.0f);
        v[j] = (a + zs) * inv;
      }
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4*>(orow + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tb, L::tcols);
  }
}

template <int KB, int VB, int D>
ChunkKernel chunk_make() {
  return ChunkKernel{chunk_attn_kernel<KB, VB, D>, ChunkSmem<D>::bytes};
}

}  // namespace kvq
