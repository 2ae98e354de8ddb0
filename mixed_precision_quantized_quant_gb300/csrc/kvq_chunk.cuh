// Causal multi-query attention over one layer's quantized cache: the queries
// of the n newest tokens attend every cached token at or before their own
// position, quantized groups dequantized and window tokens exact.  KVTuner
// (section A2, calibration design) runs prefill attention this way, over the
// dequantized cache; the attention itself is its A3 equation.
//
// Two kernels.
//
// chunk_dequant_kernel<KB, VB, D> unpacks each 64-token tile of a unit once
// into a workspace, already in the shared-memory layout of the MMA operands:
//   keys   k^ = code*s + z in fp32, split into fp16 hi + lo halves (so the
//          products keep about 22 bits), K-major core matrices;
//   values codes as exact fp16 integers (the window's values as they are),
//          token-major, the MN-major form of the P.V product's B operand;
//   the per-token value (scale, zero); window tokens (1, 0).
// Tiles cover the quantized groups [0, n_q) in steps of 64, then the FP16
// window [n_q, T) in steps of 64; tokens past a region's end are zero.
//
// chunk_attn_kernel<D>: one CTA owns 256 (query, head) rows of one (batch,
// kv head) unit, as two groups of 128 rows (one MMA tile, M = 128, each; one
// softmax thread per row), plus one warp whose first thread copies tiles in
// (bulk copies, two stages, keys and values released separately) and issues
// every tensor-core MMA:
//   S = Q K^T  (hi, then lo) into tensor memory, 64 fp32 columns per group,
//              double-buffered so that the scores of tile it+1 run while the
//              softmax of tile it does;
//   O += P' C  (hi, then lo) into tensor memory, d fp32 columns per group.
// Each softmax thread loads its row of S, runs the online softmax in the log2
// domain (lazy rescale of O when the max grows by more than 2^8), writes
// P' = p * s_value as fp16 hi + lo rows and keeps l = sum p and zs = sum p z
// in registers, so the value zero never enters an MMA.  The epilogue returns
// (O + zs) / l.  3-bit value rows store their 2-bit field (channel 11w + 10)
// with scale s2 = (7 s)/3; those codes enter C as 7 * code, and their O
// columns are divided by 3 once before the window tiles (or at the end).
#pragma once

#include <cuda_fp16.h>

#include "kvq_kernels.h"
#include "kvq_tc.cuh"

namespace kvq {

constexpr int kChunkRows = 256;                        // (query, head) rows per CTA: two groups
constexpr int kChunkM = 128;                           // rows per group: the MMA's M
constexpr int kChunkTile = 64;                         // tokens per tile
constexpr int kChunkThreads = 256;                     // softmax threads, one per row
constexpr int kChunkCtaThreads = kChunkThreads + 64;   // the copy + score-MMA warp, the P.V-MMA warp
constexpr int kDequantThreads = 256;

// One dequantized tile, in the workspace and (copied verbatim) in shared
// memory: [K hi][K lo][V], each [64 tokens][D] f16 core-matrix tiles, then 64
// (scale, zero) f16 pairs.  Keys and values are copied separately.
template <int D>
struct ChunkTile {
  static constexpr int KC = D / 8;
  static constexpr uint32_t kh = 0;
  static constexpr uint32_t kl = kChunkTile * D * 2;
  static constexpr uint32_t v = 2 * kChunkTile * D * 2;
  static constexpr uint32_t sz = 3 * kChunkTile * D * 2;
  static constexpr uint32_t kbytes = 2 * kChunkTile * D * 2;              // keys, one bulk copy
  static constexpr uint32_t vbytes = kChunkTile * D * 2 + kChunkTile * 4;  // values + pairs, one bulk copy
  static constexpr uint32_t bytes = kbytes + vbytes;
};

template <int D>
struct ChunkSmem {
  using T = ChunkTile<D>;
  static constexpr int KC = D / 8;
  static constexpr uint32_t q = 0;                                  // [256 rows][D] f16
  static constexpr uint32_t stage = q + kChunkRows * D * 2;         // two tile buffers
  static constexpr uint32_t ph = stage + 2 * T::bytes;              // [256 rows][64 tokens] f16, hi
  static constexpr uint32_t pl = ph + kChunkRows * kChunkTile * 2;  // lo
  static constexpr uint32_t pgroup = kChunkM * kChunkTile * 2;      // bytes of one group's P
  static constexpr uint32_t bars = pl + kChunkRows * kChunkTile * 2;  // 20 mbarriers
  static constexpr uint32_t tslot = bars + 192;                     // tensor-memory address
  static constexpr uint32_t bytes = tslot + 16;
  // tensor memory: S of buffer b, group g in columns [64 (2b + g), +64); O of
  // group g in [256 + D g, +D)
  static constexpr uint32_t tcols = 512;
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

// exact small integer code (< 1024) as fp32: 2^23 + code, minus 2^23
__device__ __forceinline__ float code_f32(uint32_t c) { return __uint_as_float(0x4B000000u | c) - 8388608.0f; }

// ---------------------------------------------------------------------------
// Unpack tile `blockIdx.x` of unit `blockIdx.y` into the workspace.
template <int KB, int VB, int D>
__global__ void __launch_bounds__(kDequantThreads) chunk_dequant_kernel(ChunkParams p) {
  using T = ChunkTile<D>;
  constexpr int KC = T::KC;
  constexpr int kTile = kChunkTile;
  const int tid = threadIdx.x;
  const int u = blockIdx.y, tile = blockIdx.x;
  const int gs = p.gshift;  // G = 1 << gs
  const int ntq = (p.n_q + kTile - 1) / kTile;
  const bool quant = tile < ntq;
  const int t0 = quant ? tile * kTile : p.n_q + (tile - ntq) * kTile;
  const int tq_end = quant ? min(t0 + kTile, p.n_q) : min(t0 + kTile, p.T);  // tokens that exist
  const uint8_t* urec = p.records + static_cast<int64_t>(u) * p.unit_rec_stride;
  uint8_t* dst = p.ws + (static_cast<int64_t>(u) * p.ws_tiles + tile) * T::bytes;
  if (!in_range(dst, T::bytes, p.ws, p.ws_hi, p.err)) return;  // debug builds (uniform over the CTA)

  // Thread (tid & 7) fills row tid & 7 of every core matrix it touches (8
  // consecutive threads write one whole 128-byte core matrix); its channel
  // octet kc is fixed and its tokens are row0 + kStep * j.
  constexpr int kJ = kTile * KC / kDequantThreads;
  constexpr int kStep = kDequantThreads / KC;
  const int kc = (tid >> 3) & (KC - 1);
  const int c0 = kc * 8;
  const int row0 = (tid & 7) + 8 * (tid / (8 * KC));
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);

  if (quant) {
    Unpack8<KB> ku;
    Unpack8<VB> vu;
    ku.init(c0);
    vu.init(c0);
    const int voff = p.G * p.wk;  // value code rows follow the key code rows
    // all loads of the tile first
    uint32_t kw0[kJ], kw1[kJ], vw0[kJ], vw1[kJ];
    __half2 ksz[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int t = t0 + row0 + kStep * j;
      kw0[j] = kw1[j] = vw0[j] = vw1[j] = 0u;
      ksz[j] = __floats2half2_rn(0.0f, 0.0f);
      if (t < tq_end) {
        const int gi = t >> gs, rr = t - (gi << gs);
        const uint8_t* rec = urec + static_cast<int64_t>(gi) * p.rec_bytes;
        if (!in_range(rec, p.rec_bytes, p.buf_lo, p.buf_hi, p.err)) continue;  // debug builds
        const uint32_t* krow = reinterpret_cast<const uint32_t*>(rec) + rr * p.wk;
        const uint32_t* vrow = reinterpret_cast<const uint32_t*>(rec) + voff + rr * p.wv;
        const int xk = code_word_xor(p.wk, true, rr), xv = code_word_xor(p.wv, false, rr);
        kw0[j] = krow[ku.wa ^ xk];
        if (ku.second_word()) kw1[j] = krow[(ku.wa + 1) ^ xk];
        vw0[j] = vrow[vu.wa ^ xv];
        if (vu.second_word()) vw1[j] = vrow[(vu.wa + 1) ^ xv];
        if (p.km) ksz[j] = *reinterpret_cast<const __half2*>(rec + p.off_kscale + rr * 4);
      }
    }
    // per-channel key (scale, zero) of the (at most two) groups of the
    // thread's tokens, both below n_q / G
    float sA[8], zA[8], sB[8], zB[8];
    const int gA = min(t0 + row0, tq_end - 1) >> gs;
    const int gB = min(t0 + row0 + kStep * (kJ - 1), tq_end - 1) >> gs;
    if (p.km == 0) {
      const uint8_t* recA = urec + static_cast<int64_t>(gA) * p.rec_bytes + p.off_kscale;
      const uint8_t* recB = urec + static_cast<int64_t>(gB) * p.rec_bytes + p.off_kscale;
      if (!in_range(recA, 4 * D, p.buf_lo, p.buf_hi, p.err) || !in_range(recB, 4 * D, p.buf_lo, p.buf_hi, p.err))
        return;  // debug builds
      const int cs = KB == 3 ? c0 : kscale_pos(c0, D);  // (c0 starts an 8-channel chunk)
      const uint4 sa = *reinterpret_cast<const uint4*>(recA + cs * 2);
      const uint4 za = *reinterpret_cast<const uint4*>(recA + D * 2 + cs * 2);
      const uint4 sb = *reinterpret_cast<const uint4*>(recB + cs * 2);
      const uint4 zb = *reinterpret_cast<const uint4*>(recB + D * 2 + cs * 2);
      const __half* psa = reinterpret_cast<const __half*>(&sa);
      const __half* pza = reinterpret_cast<const __half*>(&za);
      const __half* psb = reinterpret_cast<const __half*>(&sb);
      const __half* pzb = reinterpret_cast<const __half*>(&zb);
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
      const bool inB = (t >> gs) != gA;
      const uint32_t k0 = KB == 2 ? (kw0[j] >> ku.sh0) : kw0[j];
      const uint32_t v0 = VB == 2 ? (vw0[j] >> vu.sh0) : vw0[j];
      uint32_t hw[4], lw[4], vh[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        float kv[2];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          float sc, zc;
          if (p.km == 0) {
            sc = inB ? sB[e + q2] : sA[e + q2];
            zc = inB ? zB[e + q2] : zA[e + q2];
          } else {
            const float2 sz = __half22float2(ksz[j]);
            sc = sz.x;
            zc = sz.y;
            if constexpr (KB == 3) {
              if ((ku.two >> (e + q2)) & 1u) sc = __fdiv_rn(__fmul_rn(sc, 7.0f), 3.0f);
            }
          }
          kv[q2] = fmaf(code_f32(ku.get(k0, kw1[j], e + q2)), sc, zc);
        }
        split_hi_lo(kv[0], kv[1], hw[e / 2], lw[e / 2]);
        // value codes (< 1024) as exact fp16 integers: (1024 + code) - 1024
        uint32_t c_lo = vu.get(v0, vw1[j], e), c_hi = vu.get(v0, vw1[j], e + 1);
        if constexpr (VB == 3) {
          if ((vu.two >> e) & 1u) c_lo *= 7u;
          if ((vu.two >> (e + 1)) & 1u) c_hi *= 7u;
        }
        const uint32_t mag = 0x64006400u | c_lo | (c_hi << 16);
        vh[e / 2] = h2_as_u32(__hsub2(u32_as_h2(mag), __float2half2_rn(1024.0f)));
      }
      const bool live = t < tq_end;
      const uint32_t off = core_off(nn, c0, KC);
      *reinterpret_cast<uint4*>(dst + T::kh + off) = live ? make_uint4(hw[0], hw[1], hw[2], hw[3]) : zero;
      *reinterpret_cast<uint4*>(dst + T::kl + off) = live ? make_uint4(lw[0], lw[1], lw[2], lw[3]) : zero;
      *reinterpret_cast<uint4*>(dst + T::v + off) = live ? make_uint4(vh[0], vh[1], vh[2], vh[3]) : zero;
    }
    if (tid < kTile) {
      const int t = t0 + tid;
      __half2 sz = __floats2half2_rn(0.0f, 0.0f);
      if (t < tq_end) {
        const int gi = t >> gs, rr = t - (gi << gs);
        sz = *reinterpret_cast<const __half2*>(urec + static_cast<int64_t>(gi) * p.rec_bytes + p.off_vsz + rr * 4);
      }
      *reinterpret_cast<__half2*>(dst + T::sz + tid * 4) = sz;
    }
  } else {
    const __half* rk = p.res_k + static_cast<int64_t>(u) * p.res_stride;
    const __half* rv = p.res_v + static_cast<int64_t>(u) * p.res_stride;
    uint4 kr[kJ], vr[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int t = t0 + row0 + kStep * j;
      kr[j] = vr[j] = zero;
      if (t < tq_end) {
        const int slot = t % p.R;
        const int64_t off = static_cast<int64_t>(slot) * D + ((kc ^ (slot & 7)) * 8);
        if (!in_range(rk + off, 16, p.buf_lo, p.buf_hi, p.err) || !in_range(rv + off, 16, p.buf_lo, p.buf_hi, p.err))
          continue;  // debug builds
        kr[j] = *reinterpret_cast<const uint4*>(rk + off);
        vr[j] = *reinterpret_cast<const uint4*>(rv + off);
      }
    }
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const uint32_t off = core_off(row0 + kStep * j, c0, KC);
      *reinterpret_cast<uint4*>(dst + T::kh + off) = kr[j];
      *reinterpret_cast<uint4*>(dst + T::kl + off) = zero;
      *reinterpret_cast<uint4*>(dst + T::v + off) = vr[j];
    }
    if (tid < kTile)
      *reinterpret_cast<__half2*>(dst + T::sz + tid * 4) =
          __floats2half2_rn(t0 + tid < tq_end ? 1.0f : 0.0f, 0.0f);
  }
}

// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kChunkCtaThreads, 1) chunk_attn_kernel(ChunkParams p) {
  using L = ChunkSmem<D>;
  using T = ChunkTile<D>;
  constexpr int KC = L::KC;
  constexpr int kTile = kChunkTile;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* kfull = reinterpret_cast<uint64_t*>(sm + L::bars);  // [stage]: keys landed (tx)
  uint64_t* vfull = kfull + 2;   // [stage]: values and pairs landed (tx)
  uint64_t* kfree = kfull + 4;   // [stage]: the scores that read the keys are done (commit)
  uint64_t* vfree = kfull + 6;   // [stage]: the P.V products that read the values are done (commit)
  uint64_t* s_done = kfull + 8;  // [stage][group]: scores ready (commit)
  uint64_t* p_full = kfull + 12; // [group]: P' written, O rescaled (128 arrivals)
  uint64_t* o_done = kfull + 14; // [group]: P.V done (commit)
  uint64_t* s_free = kfull + 16; // [stage][group]: the group's rows have read their scores (128 arrivals)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::tslot);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int grp = (tid >> 7) & 1;  // row group of a softmax thread

  const int u = blockIdx.y;
  const int blk = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);  // longest rows first
  const int b = u / p.kv_heads, hk = u - b * p.kv_heads;
  const int i0 = blk * p.qpb;
  const int nqb = min(p.qpb, p.n - i0);
  const int rows = nqb * p.gqa;
  const int pos0 = p.T - p.n;  // position of query 0
  const int last_pos = pos0 + i0 + nqb - 1;
  const uint8_t* wsu = p.ws + static_cast<int64_t>(u) * p.ws_tiles * T::bytes;

  // ---- query rows -> shared memory (row r = query r / gqa, head r % gqa)
  if (tid < kChunkThreads) {
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
  }
  if (tid == 0) {
    for (int i = 0; i < 12; ++i) mbar_init(kfull + i, 1);
    mbar_init(p_full, kChunkM);
    mbar_init(p_full + 1, kChunkM);
    mbar_init(o_done, 1);
    mbar_init(o_done + 1, 1);
    for (int i = 0; i < 4; ++i) mbar_init(s_free + i, kChunkM);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, L::tcols);
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = *tslot;

  const int endQ = min(p.n_q, last_pos + 1);
  const int ntq = (endQ + kTile - 1) / kTile;
  const int endW = last_pos + 1;
  const int ntw = endW > p.n_q ? (endW - p.n_q + kTile - 1) / kTile : 0;
  const int ntiles = ntq + ntw;  // the unit's tiles 0 .. ntiles-1 (same numbering as the workspace)

  if (warp >= kChunkThreads / 32) {
    // ================= MMA warps.  The first thread of warp 8 issues every
    // bulk copy and the score MMAs: per tile it, S(it) (once the rows have
    // read S(it-2) from the same buffer); the keys of tile it+1 into the other
    // stage (freed by S(it-1)); the values and pairs of tile it into its stage
    // (freed by P.V(it-2)).  The first thread of warp 9 issues the P.V MMAs
    // of each tile once its softmax is done, so the two MMA streams are
    // issued by different warps.
    const bool score_warp = warp == kChunkThreads / 32;
    if ((tid & 31) == 0) {
      const uint32_t sq = smem_u32(sm + L::q);
      const uint32_t sst = smem_u32(sm + L::stage);
      const uint32_t sph = smem_u32(sm + L::ph), spl = smem_u32(sm + L::pl);
      constexpr uint32_t idS = idesc_f16_f32(kChunkM, kTile);
      constexpr uint32_t idO = idesc_f16_f32(kChunkM, D) | (1u << 16);  // B (values) MN-major
      // (debug builds: a source outside the workspace is recorded and skipped;
      // the barrier still completes)
      auto copy_k = [&](int it) {
        uint64_t* bar = kfull + (it & 1);
        const uint8_t* src = wsu + static_cast<int64_t>(it) * T::bytes;
        if (!in_range(src, T::kbytes, p.ws, p.ws_hi, p.err)) {
          mbar_arrive(bar);
          return;
        }
        mbar_arrive_expect_tx(bar, T::kbytes);
        bulk_g2s(sm + L::stage + (it & 1) * T::bytes, src, T::kbytes, bar);
      };
      auto copy_v = [&](int it) {
        uint64_t* bar = vfull + (it & 1);
        const uint8_t* src = wsu + static_cast<int64_t>(it) * T::bytes + T::v;
        if (!in_range(src, T::vbytes, p.ws, p.ws_hi, p.err)) {
          mbar_arrive(bar);
          return;
        }
        mbar_arrive_expect_tx(bar, T::vbytes);
        bulk_g2s(sm + L::stage + (it & 1) * T::bytes + T::v, src, T::vbytes, bar);
      };
      auto issue_pv = [&](int it, bool& bad) {
        const int bs = it & 1;
        bad = bad || !mbar_wait(vfull + bs, (it >> 1) & 1, p.err);
        const uint32_t vb_ = sst + bs * T::bytes + T::v;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          bad = bad || !mbar_wait(p_full + g, it & 1, p.err);
          if (bad) return;
          tc_fence_after_sync();
          const uint32_t dO = tb + 4 * kTile + D * g;
          const uint32_t pg = g * L::pgroup;
          // descriptors of k-step 0; a k-step moves the address field (bytes / 16)
          const uint64_t dph = smem_desc(sph + pg, 128, (kTile / 8) * 128);
          const uint64_t dpl = smem_desc(spl + pg, 128, (kTile / 8) * 128);
          const uint64_t dv = smem_desc(vb_, KC * 128, 128);
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            umma_f16(dO, dph + 16 * ks, dv + 2 * KC * 8 * ks, idO, (it > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) umma_f16(dO, dpl + 16 * ks, dv + 2 * KC * 8 * ks, idO, 1u);
          umma_commit(o_done + g);
        }
        umma_commit(vfree + bs);
      };
      bool bad = false;
      if (!score_warp) {
#pragma unroll 1
        for (int it = 0; it < ntiles && !bad; ++it) issue_pv(it, bad);
      } else {
      copy_k(0);
      copy_v(0);
#pragma unroll 1
      for (int it = 0; it < ntiles && !bad; ++it) {
        const int bs = it & 1;
        bad = !mbar_wait(kfull + bs, (it >> 1) & 1, p.err);
        if (bad) break;
        tc_fence_after_sync();
        const uint32_t kb_h = sst + bs * T::bytes, kb_l = kb_h + T::kl;
        // both groups' rows have read S(it-2), the buffer's previous scores
        if (it >= 2) {
          bad = !mbar_wait(s_free + 2 * bs, ((it - 2) >> 1) & 1, p.err);
          bad = bad || !mbar_wait(s_free + 2 * bs + 1, ((it - 2) >> 1) & 1, p.err);
        }
        if (bad) break;
        tc_fence_after_sync();
        {
          // the two groups' accumulation chains alternate: an MMA whose
          // accumulator the previous MMA writes waits for it, one into the
          // other group's columns need not
          const uint32_t dS0 = tb + kTile * (2 * bs), dS1 = dS0 + kTile;
          const uint64_t dq0 = smem_desc(sq, 128, KC * 128), dq1 = smem_desc(sq + kChunkM * D * 2, 128, KC * 128);
          const uint64_t dkh = smem_desc(kb_h, 128, KC * 128), dkl = smem_desc(kb_l, 128, KC * 128);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            umma_f16(dS0, dq0 + 16 * ks, dkh + 16 * ks, idS, ks > 0);
            umma_f16(dS1, dq1 + 16 * ks, dkh + 16 * ks, idS, ks > 0);
          }
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            umma_f16(dS0, dq0 + 16 * ks, dkl + 16 * ks, idS, 1u);
            umma_f16(dS1, dq1 + 16 * ks, dkl + 16 * ks, idS, 1u);
          }
          umma_commit(s_done + 2 * bs);
          umma_commit(s_done + 2 * bs + 1);
        }
        umma_commit(kfree + bs);
        // keys of tile it+1 into the other stage (its scores of tile it-1 are long done)
        if (it + 1 < ntiles) {
          if (it >= 1) bad = !mbar_wait(kfree + (bs ^ 1), ((it - 1) >> 1) & 1, p.err);
          if (bad) break;
          copy_k(it + 1);
        }
        // values and pairs of tile it (tile 0's were copied first); the stage's
        // P.V of tile it-2 was issued an iteration ago
        if (it >= 1) {
          if (it >= 2) bad = !mbar_wait(vfree + bs, ((it - 2) >> 1) & 1, p.err);
          if (bad) break;
          copy_v(it);
        }
      }
      // copies still in flight (only after a failed wait) must land before exit
      if (bad) {
        mbar_wait(kfull, 0, p.err, 1u << 16);
        mbar_wait(vfull, 0, p.err, 1u << 16);
      }
      }
    }
    __syncwarp();
  } else {
    // ================= softmax threads (one row each)
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tb + kTile * grp + lane_off;          // + 2 kTile for S buffer 1
    const uint32_t tO = tb + 4 * kTile + D * grp + lane_off;  // this warp's lanes of O
    const int r = tid;
    const int lim = (r < rows) ? pos0 + i0 + r / p.gqa : last_pos;
    float m = -INFINITY, l = 0.0f, zs = 0.0f;
    bool failed = false;
    uint8_t* prow_h = sm + L::ph + grp * L::pgroup;
    uint8_t* prow_l = sm + L::pl + grp * L::pgroup;

#pragma unroll 1
    for (int it = 0; it < ntiles; ++it) {
      const bool quant = it < ntq;
      const int t0 = quant ? it * kTile : p.n_q + (it - ntq) * kTile;
      const int tend = quant ? min(t0 + kTile, endQ) : min(t0 + kTile, endW);
      const int bs = it & 1;
      // scores of tile it, its values' pairs, and this group's P.V of tile it-1 (P and O reuse)
      if (!failed) failed = !mbar_wait(s_done + 2 * bs + grp, (it >> 1) & 1, p.err);
      if (!failed) failed = !mbar_wait(vfull + bs, (it >> 1) & 1, p.err);
      if (it >= 1 && !failed) failed = !mbar_wait(o_done + grp, (it - 1) & 1, p.err);
      tc_fence_after_sync();
      const uint32_t tSb = tS + 2 * kTile * bs;
      const __half2* szr = reinterpret_cast<const __half2*>(sm + L::stage + bs * T::bytes + T::sz);

      // ---- online softmax of this thread's row: its 64 scores come from
      // tensor memory in one batch of loads (a single wait)
      // tokens t0 .. t0 + nvis - 1 are visible to this row
      const int nvis = min(tend, lim + 1) - t0;
      const bool full = __all_sync(0xffffffffu, nvis >= kTile);
      uint32_t x0[16], x1[16], x2[16], x3[16];
      tmem_ld16(tSb, x0);
      tmem_ld16(tSb + 16, x1);
      tmem_ld16(tSb + 32, x2);
      tmem_ld16(tSb + 48, x3);
      tmem_ld_wait(x0);  // waits for all four
      tmem_ld_wait(x1);
      tmem_ld_wait(x2);
      tmem_ld_wait(x3);
      tc_fence_before_sync();
      mbar_arrive(s_free + 2 * bs + grp);  // S buffer bs may take tile it+2
      auto score = [&](int j) -> float {
        const uint32_t v = j < 16 ? x0[j] : j < 32 ? x1[j - 16] : j < 48 ? x2[j - 32] : x3[j - 48];
        return (full || j < nvis) ? __uint_as_float(v) : -INFINITY;
      };
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTile; ++j) mx = fmaxf(mx, score(j));
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
      const bool third = p.vb == 3 && it == ntq && ntq > 0;
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
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int jj = 32 * half + j;
          const float2 sz0 = __half22float2(szr[jj]), sz1 = __half22float2(szr[jj + 1]);
          const float p0 = ex2(fmaf(score(jj), p.alpha, nm));
          const float p1 = ex2(fmaf(score(jj + 1), p.alpha, nm));
          ls += p0 + p1;
          zsum = fmaf(p0, sz0.y, fmaf(p1, sz1.y, zsum));
          split_hi_lo(p0 * sz0.x, p1 * sz1.x, hi[j / 2], lo[j / 2]);
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t off = core_off(r & 127, 32 * half + 8 * cc, kTile / 8);
          *reinterpret_cast<uint4*>(prow_h + off) = make_uint4(hi[4 * cc], hi[4 * cc + 1], hi[4 * cc + 2], hi[4 * cc + 3]);
          *reinterpret_cast<uint4*>(prow_l + off) = make_uint4(lo[4 * cc], lo[4 * cc + 1], lo[4 * cc + 2], lo[4 * cc + 3]);
        }
      }
      l += ls;
      zs += zsum;
      // P' visible to the tensor core, TMEM reads and the O rescale ordered
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(p_full + grp);
    }

    // ---- epilogue: out = (O + zs) / l
    if (!failed && ntiles > 0) failed = !mbar_wait(o_done + grp, (ntiles - 1) & 1, p.err);
    tc_fence_after_sync();
    const bool third = p.vb == 3 && ntw == 0;
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
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tb, L::tcols);
  }
}

template <int KB, int VB, int D>
ChunkDequant chunk_dequant_make() {
  return ChunkDequant{chunk_dequant_kernel<KB, VB, D>};
}

}  // namespace kvq
