// Fused decode attention over a layer of the mixed-precision KV cache:
// unpack -> dequantize -> q.K^T -> online softmax -> .V, split over the
// context with an in-kernel merge.
//
// a = softmax(q K^T / sqrt(d)), o = a V with K, V the concatenation of the
// quantized groups (dequantized on the fly) and the FP16 residual window
// ("KVTuner ...", section A3 equation; "KVmix ...", 关键设计 4: dequantize on the
// fly and multiply with the query in one kernel).
//
// Work decomposition: the flat list of work items (per (batch, kv head) unit:
// its quantized groups, then its residual window in tiles of 16 tokens) is cut
// into equal-byte ranges, one per CTA of a single wave.  Inside a CTA each
// warp takes every fourth item and streams it into shared memory with a 1-D
// bulk TMA copy (warp-private stages, mbarrier completion, bounded waits).
// All query heads of a kv head are processed together.
//
// Arithmetic (all exact except the fp32 accumulation and exp2):
//   * codes become exact fp16 integers with the 1024-exponent trick;
//   * the per-channel key scale is folded into the query: q~_c = q_c * s_c,
//     split into fp16 hi + lo parts that sit in separate MMA columns; the
//     per-channel zero contributes sum_c q_c z_c, computed by one extra MMA per
//     group with the zeros broadcast over the rows;
//   * the per-token value scale is folded into the probabilities:
//     p~_t = p_t * s_t (hi + lo columns); the value zero adds sum_t p_t z_t;
//   * mma.sync m16n8k16 (fp16 in, fp32 accumulate): for q.K^T the rows are 16
//     tokens and the columns 4 query heads x (hi, lo); for p.V the rows are 16
//     channels and the reduction runs over the 16 tokens.
// The residual window is read with ldmatrix from chunk-swizzled rows.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

constexpr int kSlice = 32;   // tokens of a key group one warp takes per stage
constexpr int kStages = 2;   // CTA-wide stages in flight

// Bytes one 32-token slice of a group record stands for: [K rows][V rows]
// then [K scale d][K zero d] (per-channel keys) or [K (scale, zero) 32 pairs]
// (per-token keys), then [V (scale, zero) 32 pairs].
__host__ __device__ constexpr int slice_bytes(int D, int wk, int wv, int km) {
  return kSlice * 4 * (wk + wv) + (km ? 4 * kSlice : 4 * D) + 4 * kSlice;
}

// Bytes of one stage: W/NS whole key-group records (W slices; their bytes
// are at most W slice_bytes for any G), or as many residual window tiles as
// fit, at least one.
__host__ __device__ constexpr int stage_bytes(int D, int cq, int W) {
  const int rt = kResTile * 4 * D;
  const int need = (rt > W * cq) ? rt : W * cq;
  return (need + 127) / 128 * 128;
}

struct DecodeSmem {
  int stage;
  int off_bars, off_cnt, off_qs, off_qp, off_qps, off_qr, off_qsum, off_wm, off_wl, off_dm, off_flags, off_wo, total;
};

// kStages stages of `stage` bytes shared by the CTA's W warps, then the
// barriers, the query rows and tables, and the per-warp merge area.
__host__ __device__ constexpr DecodeSmem decode_smem_layout_stage(int D, int NT, int stage, int W) {
  DecodeSmem s{};
  const int H = 4 * NT;
  s.stage = stage;
  int off = kStages * stage;
  s.off_bars = off;
  off += (kStages + 2) * 8;          // stage fills, then the two query buffers
  s.off_cnt = off;
  off += 16;                         // per stage: warps done with it, over all fills
  s.off_qs = off;
  off += 2 * H * D * 2;              // double-buffered query rows of a unit
  // per-lane query tables, lane-interleaved in 8-byte pairs (conflict-free)
  s.off_qp = off;
  off += 32 * NT * 18 * 4;           // key-pair query table (up to 18 pairs per thread)
  s.off_qps = off;
  off += 32 * NT * 18 * 4;           // same, scaled by 2^(Pmax - pos) per pair
  s.off_qr = off;
  off += 32 * NT * D / 16 * 2 * 4;   // residual (fp16 key) query table
  s.off_qsum = off;
  off += H * 4;                      // per head sum of the query (per-token keys)
  s.off_wm = off;
  off += W * H * 4;
  s.off_wl = off;
  off += W * H * 4;
  s.off_dm = off;
  off += W * H * 4;
  s.off_flags = off;
  off += 64;
  off = (off + 15) / 16 * 16;
  s.off_wo = off;
  off += W * H * D * 4;
  s.total = off;
  return s;
}

__host__ __device__ inline DecodeSmem decode_smem_layout(int D, int NT, int cq, int W) {
  return decode_smem_layout_stage(D, NT, stage_bytes(D, cq, W), W);
}

// Word of channel ch of head h inside a warp's partial-output rows: ch XOR a
// 5-bit key of (h, ch / 32), a permutation within each 32-channel block, so
// the merge still reads 32 consecutive channels from 32 banks.  The keys
// spread the epilogue's stores over the banks: the 8-head form stores, per
// instruction, one channel offset for all (head g, lane column tig) and the
// key (g bits 0, 3, 4; tig = block bits 1, 2) tells the 32 lanes apart; the
// 1-4-head form stores channel 16g + mt of head 4j + tig and the key (tig
// bits 2, 3; block bits 0, 1) does the same with the channel's own bit 4.
template <bool kT>
__device__ __forceinline__ int wo_chan(int h, int ch) {
  const int b = ch >> 5;
  const int key = kT ? (((h & 1) | ((h >> 1) << 3)) ^ (b << 1)) : (((h & 3) << 2) | (b & 3));
  return ch ^ (key & 31);
}

// Warps per CTA of an instantiation: 8 where two such CTAs fit in an SM's
// shared memory (fewer CTAs per unit: fewer query-table builds and split
// merges at the same occupancy), else 4.  3-bit values keep 4: they need more
// than the 128 registers a thread may use at 2 x 256 threads per SM.  The
// stage size does not depend on G.
template <int KB, int VB, int D, int NT, int KM>
__host__ __device__ constexpr int decode_warps() {
  constexpr int WK = (KB == 3) ? (D + 10) / 11 : D * KB / 32;
  constexpr int WV = (VB == 3) ? (D + 10) / 11 : D * VB / 32;
  constexpr int cq = slice_bytes(D, WK, WV, KM);
  constexpr int smem8 = decode_smem_layout_stage(D, NT, stage_bytes(D, cq, 8), 8).total;
  return (NT == 1 && VB != 3 && 2 * (smem8 + 1024) <= 228 * 1024) ? 8 : 4;
}

// ------------------------------------------------------------------ unpacking

template <int N>
__device__ __forceinline__ void lds_words(uint32_t (&w)[N], const uint32_t* p);

// N words w0 .. w0 + N - 1 of a code row stored with word-index XOR xm (xm
// moves whole 4-word groups, or N-word groups when N < 4)
template <int N>
__device__ __forceinline__ void lds_row_words(uint32_t (&w)[N], const uint32_t* row, int w0, int xm) {
  if constexpr (N < 4) {
    lds_words<N>(w, row + (w0 ^ xm));
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + ((w0 + i) ^ xm));
      w[i] = v.x;
      w[i + 1] = v.y;
      w[i + 2] = v.z;
      w[i + 3] = v.w;
    }
  }
}

template <int N>
__device__ __forceinline__ void lds_words(uint32_t (&w)[N], const uint32_t* p) {
  if constexpr (N == 1) {
    w[0] = p[0];
  } else if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x;
    w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(p + i);
      w[i] = v.x;
      w[i + 1] = v.y;
      w[i + 2] = v.z;
      w[i + 3] = v.w;
    }
  }
}

// Score k-steps (pairs of channels per thread per token row = 2 x this).
// 3-bit keys: each thread owns 3 (d128) or 2 (d64) words of 11 fields.
template <int KB, int D>
struct KeyShape {
  static constexpr int WK = (KB == 3) ? (D + 10) / 11 : D * KB / 32;  // words per token row
  static constexpr int WT = (KB == 3) ? (D == 128 ? 3 : 2) : WK / 4;  // words per thread
  static constexpr int KSK = (KB == 3) ? (D == 128 ? 9 : 6) : D / 16;
  static constexpr int NPK = 2 * KSK;
  static constexpr int PW = (KB == 3) ? 5 : 16 / KB;                  // pairs per word
};

// Value m-tiles in the quantized-path channel map (3-bit adds a tile for the
// 2-bit fields of the 11-field words).
template <int VB, int D>
struct ValShape {
  static constexpr int WV = (VB == 3) ? (D + 10) / 11 : D * VB / 32;
  static constexpr int MT3 = (D == 128) ? 8 : 5;
  static constexpr int MTV = (VB == 3) ? MT3 + 1 : D / 16;
  static constexpr int VW = (VB == 3) ? 1 : ((D * VB / 256) > 0 ? (D * VB / 256) : 1);
};

// Codes enter the tensor cores as exact fp16 subnormals: a field masked in
// place at bit position pos (pos + width <= 10) is the fp16 value
// code * 2^(pos - 24).  The power-of-two factor is removed outside the MMA:
// for keys it is folded into the query column of that k-slot (q scaled by
// 2^(Pmax - pos), so every product carries 2^(Pmax - 24)); for values every
// row of a value m-tile shares one position and the fp32 accumulator of that
// tile is rescaled once at the end.

// Channels (ca, cb) of key pair pi of thread tig (-1 for padding).
//  4-bit: (c0,c4) (c1,c5) (c2,c6) (c3,c7) per word; 2-bit: (c_i, c_{8+i});
//  8-bit: (c0,c2) (c1,c3); 3-bit: fields (i, i+5) of each word, then the
//  2-bit fields of the thread's words paired two by two.
template <int KB, int D>
__device__ __forceinline__ void key_pair_channels(int tig, int pi, int& ca, int& cb) {
  using S = KeyShape<KB, D>;
  if constexpr (KB == 3) {
    const int w0 = tig * S::WT;
    if (pi < 5 * S::WT) {
      const int base = 11 * (w0 + pi / 5);
      ca = base + pi % 5;
      cb = ca + 5;
    } else {
      const int k = pi - 5 * S::WT;
      ca = (2 * k < S::WT) ? 11 * (w0 + 2 * k) + 10 : -1;
      cb = (2 * k + 1 < S::WT) ? 11 * (w0 + 2 * k + 1) + 10 : -1;
    }
    if (ca >= D) ca = -1;
    if (cb >= D) cb = -1;
  } else {
    const int wi = pi / S::PW, e = pi % S::PW;
    const int cbase = tig * (D / 4) + wi * (32 / KB);
    ca = cbase + e;
    cb = cbase + e + (KB == 4 ? 4 : (KB == 2 ? 8 : 2));
  }
}

// Bit position of key pair pi inside its 16-bit half, and the largest one.
template <int KB, int D>
__host__ __device__ constexpr int key_pos(int pi) {
  if (KB == 4) return 4 * (pi & 1);
  if (KB == 2) return 2 * (pi & 1);
  if (KB == 8) return 0;
  return (pi < 5 * KeyShape<KB, D>::WT) ? ((pi % 5) % 3) * 3 : 0;  // 3-bit: 0,3,6,0,3
}
template <int KB>
__host__ __device__ constexpr int key_pos_max() {
  return KB == 4 ? 4 : (KB == 2 ? 2 : (KB == 8 ? 0 : 6));
}

// Code pairs of one 2/4/8-bit key word in key_pair_channels order.
template <int KB>
__device__ __forceinline__ void k_word_pairs(uint32_t w, uint32_t* e) {
  if constexpr (KB == 4) {
    const uint32_t t = w >> 8;
    e[0] = w & 0x000F000Fu;
    e[1] = w & 0x00F000F0u;
    e[2] = t & 0x000F000Fu;
    e[3] = t & 0x00F000F0u;
  } else if constexpr (KB == 2) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const uint32_t t = w >> (2 * i);
      e[i] = t & 0x00030003u;
      e[i + 1] = t & 0x000C000Cu;
    }
  } else {  // 8-bit
    e[0] = prmt(w, 0u, 0x4240u);
    e[1] = prmt(w, 0u, 0x4341u);
  }
}

// Five 3-bit fields at bits 0,3,..,12 of the low halves of two words, as
// (field_i of a, field_i of b) subnormal pairs at positions 0,3,6,0,3.
__device__ __forceinline__ void lo5(uint32_t a, uint32_t b, uint32_t* e) {
  const uint32_t z = prmt(a, b, 0x5410u);
  const uint32_t z9 = z >> 9;
  e[0] = z & 0x00070007u;
  e[1] = z & 0x00380038u;
  e[2] = z & 0x01C001C0u;
  e[3] = z9 & 0x00070007u;
  e[4] = z9 & 0x00380038u;
}

// 2-bit fields (bits 30..31) of two words as one pair at position 0.
__device__ __forceinline__ uint32_t slot10_pair(uint32_t a, uint32_t b) { return prmt(a >> 30, b >> 30, 0x5410u); }

// The thread's key pairs of one token row.
template <int KB, int D>
__device__ __forceinline__ void key_row_pairs(const uint32_t* row, int tig, uint32_t* E) {
  using S = KeyShape<KB, D>;
  if constexpr (KB == 3) {
    uint32_t w[S::WT];
#pragma unroll
    for (int wi = 0; wi < S::WT; ++wi) {
      const int wd = tig * S::WT + wi;
      w[wi] = (wd < S::WK) ? row[wd] : 0u;
    }
#pragma unroll
    for (int wi = 0; wi < S::WT; ++wi) {
      // move fields 5..9 up one bit so field i and field i+5 sit 16 bits apart
      const uint32_t x = (w[wi] & 0x7FFFu) | ((w[wi] << 1) & 0xFFFF0000u);
      const uint32_t x9 = x >> 9;
      E[5 * wi + 0] = x & 0x00070007u;
      E[5 * wi + 1] = x & 0x00380038u;
      E[5 * wi + 2] = x & 0x01C001C0u;
      E[5 * wi + 3] = x9 & 0x00070007u;
      E[5 * wi + 4] = x9 & 0x00380038u;
    }
#pragma unroll
    for (int k = 5 * S::WT; k < S::NPK; ++k) {
      const int a = 2 * (k - 5 * S::WT), b = a + 1;
      E[k] = (a < S::WT) ? slot10_pair(w[a], (b < S::WT) ? w[b] : 0u) : 0u;
    }
  } else {
    uint32_t w[S::WT];
    lds_words<S::WT>(w, row + tig * S::WT);
#pragma unroll
    for (int wi = 0; wi < S::WT; ++wi) k_word_pairs<KB>(w[wi], E + wi * S::PW);
  }
}

// Value code pairs for two tokens (a, b): H[c] = (code_a[c], code_b[c]) for the
// D/8 channels this thread owns (2/4/8-bit values), as subnormals at the
// positions value_pos gives for the m-tile that uses them.
template <int VB, int D>
__device__ __forceinline__ void v_pairs(const uint32_t* wa, const uint32_t* wb, uint32_t half_sel,
                                        uint32_t (&H)[D / 8]) {
  if constexpr (VB == 2) {
    if constexpr (D == 128) {
      const uint32_t x = prmt(wa[0], wb[0], 0x5410u), y = prmt(wa[0], wb[0], 0x7632u);
      const uint32_t x10 = x >> 10, y10 = y >> 10;
#pragma unroll
      for (int i = 0; i < 5; ++i) {
        H[i] = x & (0x00030003u << (2 * i));
        H[8 + i] = y & (0x00030003u << (2 * i));
      }
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        H[5 + i] = x10 & (0x00030003u << (2 * i));
        H[13 + i] = y10 & (0x00030003u << (2 * i));
      }
    } else {
      const uint32_t x = prmt(wa[0], wb[0], half_sel);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const uint32_t t = x >> (2 * i);
        H[i] = t & 0x00030003u;
        H[i + 1] = t & 0x000C000Cu;
      }
    }
  } else if constexpr (VB == 4) {
#pragma unroll
    for (int k = 0; k < D / 64; ++k) {
      const uint32_t x = prmt(wa[k], wb[k], 0x5410u), y = prmt(wa[k], wb[k], 0x7632u);
      const uint32_t x8 = x >> 8, y8 = y >> 8;
      H[8 * k + 0] = x & 0x000F000Fu;
      H[8 * k + 1] = x & 0x00F000F0u;
      H[8 * k + 2] = x8 & 0x000F000Fu;
      H[8 * k + 3] = x8 & 0x00F000F0u;
      H[8 * k + 4] = y & 0x000F000Fu;
      H[8 * k + 5] = y & 0x00F000F0u;
      H[8 * k + 6] = y8 & 0x000F000Fu;
      H[8 * k + 7] = y8 & 0x00F000F0u;
    }
  } else {  // 8-bit
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      const uint32_t z = prmt(wa[k], wb[k], 0x5410u), y = prmt(wa[k], wb[k], 0x7632u);
      H[4 * k] = z & 0x00FF00FFu;
      H[4 * k + 1] = (z >> 8) & 0x00FF00FFu;
      H[4 * k + 2] = y & 0x00FF00FFu;
      H[4 * k + 3] = (y >> 8) & 0x00FF00FFu;
    }
  }
}

// Bit position shared by both rows of value m-tile mt (quantized channel map).
template <int VB, int D>
__host__ __device__ constexpr int value_pos(int mt) {
  if (VB == 2) return D == 128 ? 2 * (mt < 5 ? mt : mt - 5) : 2 * (mt & 1);
  if (VB == 4) return 4 * (mt & 1);
  if (VB == 8) return 0;
  // 3-bit: d128 tiles hold positions 0,0,0,3,3,3,6,6 then the 2-bit tile (0);
  // d64 tiles 0,3,6,0,3 then the 2-bit tile (0)
  if (D == 128) return mt < 3 ? 0 : (mt < 6 ? 3 : (mt < 8 ? 6 : 0));
  return mt < 5 ? ((mt % 5) % 3) * 3 : 0;
}

// Channel of row (g + 8*hi) of value m-tile mt in the quantized-path map, or -1.
//  2/4/8-bit: thread g owns channels [g*D/8, (g+1)*D/8): row g -> g*D/8 + mt,
//  row g+8 -> g*D/8 + D/16 + mt.
//  3-bit, d128: thread g owns the 3-bit fields of word g and fields
//  5h..5h+4 of word 8 + g/2 (h = g & 1).  With A = fields 0..4 of word g,
//  A' = fields 5..9 of word g and B = the owned fields of word 8 + g/2, the
//  tiles hold (row g / row g+8): A0/A3, A'0/A'3, B0/B3, A1/A4, A'1/A'4,
//  B1/B4, A2/A'2, B2/-; tile 8 holds 2-bit fields (word g, and word 8 + g/2
//  for even g while that word has one).
//  3-bit, d64: thread g < 6 owns word g: tile mt holds field mt / field 5+mt
//  (mt < 5); tile 5 holds the 2-bit field of word g < 5 in row g.
template <int VB, int D>
__device__ __forceinline__ int vq_channel(int g, int mt, int hi) {
  if constexpr (VB != 3) {
    return g * (D / 8) + (hi ? D / 16 : 0) + mt;
  } else {
    constexpr int MT3 = ValShape<VB, D>::MT3;
    if (mt == MT3) {
      if (!hi) return (D == 128 || g < 5) ? 11 * g + 10 : -1;
      if (D == 128) {
        const int wb = 8 + (g >> 1);
        return ((g & 1) == 0 && wb <= 10) ? 11 * wb + 10 : -1;
      }
      return -1;
    }
    int c;
    if (D == 128) {
      // (source, field) of each tile row: source 0 = A, 1 = A', 2 = B
      const int src_lo[8] = {0, 1, 2, 0, 1, 2, 0, 2}, fld_lo[8] = {0, 0, 0, 1, 1, 1, 2, 2};
      const int src_hi[8] = {0, 1, 2, 0, 1, 2, 1, -1}, fld_hi[8] = {3, 3, 3, 4, 4, 4, 2, 0};
      const int src = hi ? src_hi[mt] : src_lo[mt], fld = hi ? fld_hi[mt] : fld_lo[mt];
      if (src < 0) return -1;
      if (src == 0) c = 11 * g + fld;
      else if (src == 1) c = 11 * g + 5 + fld;
      else c = 11 * (8 + (g >> 1)) + 5 * (g & 1) + fld;
    } else {
      if (g >= 6) return -1;
      c = 11 * g + (hi ? 5 + mt : mt);
    }
    return c < D ? c : -1;
  }
}

__device__ __forceinline__ float reduce_over_g(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// fp16 hi + lo split of two fp32 values, as (hi pair, lo pair)
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  hi = h2_as_u32(h);
  lo = h2_as_u32(__floats2half2_rn(a - __low2float(h), b - __high2float(h)));
}

// ------------------------------------------------------------------ kernel

// KM: key mode, 0 = per channel over key groups, 1 = per token.
template <int KB, int VB, int D, int NT, int KM>
__global__ void __launch_bounds__(32 * decode_warps<KB, VB, D, NT, KM>(),
                                  decode_warps<KB, VB, D, NT, KM>() == 8 ? 2 : 3)
    decode_kernel(DecodeParams p) {
  static_assert(KM == 0 || KB != 3, "per-token keys are 2, 4 or 8 bits");
  using KS_ = KeyShape<KB, D>;
  using VS_ = ValShape<VB, D>;
  constexpr int KS = D / 16;            // residual k-steps / channel m-tiles
  constexpr int KSK = KS_::KSK;         // quantized score k-steps
  constexpr int NPK = KS_::NPK;         // key pairs per thread per row
  constexpr int WK = KS_::WK;
  constexpr int WV = VS_::WV;
  constexpr int MTV = VS_::MTV;         // value m-tiles (quantized map)
  constexpr int MTA = MTV > KS ? MTV : KS;
  constexpr int NP = D / 8;
  constexpr int H = 4 * NT;             // padded query heads
  constexpr int W = decode_warps<KB, VB, D, NT, KM>();  // warps per CTA
  constexpr int TH = 32 * W;
  constexpr bool kTabSmem = false;
  // 5-8 query heads per kv head (2-, 4- or 8-bit codes): the 16 MMA rows are
  // the 8 heads x {hi, lo} and the tokens are the columns, so the score
  // accumulator is already the A operand of P.V (no shuffles), and the
  // query's scale fold takes two half2 operations per channel pair.
  constexpr bool kT = (NT == 2) && (KB != 3) && (VB != 3);
  constexpr int NEV = D / 8;  // P.V n-tiles of 8 channels (transposed form)

  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kCq = slice_bytes(D, WK, WV, KM);
  const DecodeSmem L = decode_smem_layout(D, NT, kCq, W);
  constexpr uint32_t SB = static_cast<uint32_t>(stage_bytes(D, kCq, W));  // bytes of one stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bars);
  __half* qs = reinterpret_cast<__half*>(smem + L.off_qs);
  uint32_t* qp_tab = reinterpret_cast<uint32_t*>(smem + L.off_qp);
  uint32_t* qps_tab = reinterpret_cast<uint32_t*>(smem + L.off_qps);
  uint32_t* qr_tab = reinterpret_cast<uint32_t*>(smem + L.off_qr);
  float* qsum_s = reinterpret_cast<float*>(smem + L.off_qsum);
  float* wm = reinterpret_cast<float*>(smem + L.off_wm);
  float* wl = reinterpret_cast<float*>(smem + L.off_wl);
  float* dm = reinterpret_cast<float*>(smem + L.off_dm);
  int* flags = reinterpret_cast<int*>(smem + L.off_flags);
  float* wo = reinterpret_cast<float*>(smem + L.off_wo);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* qtab = reinterpret_cast<uint32_t*>(wo + warp * H * D);
  int* scnt = reinterpret_cast<int*>(smem + L.off_cnt);
  const int g = lane >> 2, tig = lane & 3, part = g & 1;
  // table entry (j, pi) of lane l sits at u32 ((j*NPK + pi)/2 * 32 + l) * 2 + (pi & 1)
  auto kt_idx = [](int j, int pi, int l) { return (((j * NPK + pi) >> 1) * 32 + l) * 2 + (pi & 1); };
  auto rt_idx = [](int j, int kk, int l) { return ((j * KS + kk) * 32 + l) * 2; };

  // ---------------- state and this CTA's share of the work
  // A unit's work is a list of stages: its key groups, NR = W / NS whole
  // records per stage (one 32-token slice per warp), then its FP16 window,
  // TPS 16-token tiles per stage.  The flat list of stages (unit by unit) is
  // cut into P near-equal cost ranges, x(p) = p*floor(C/P) + min(p, C mod P);
  // each unit also carries a fixed cost for its setup and merge, so CTAs that
  // span two units get fewer bytes.  A stage belongs to the CTA whose range
  // holds its start.  All of it is 32-bit arithmetic (the host keeps a
  // layer's decode bytes below 2^32), computed by every thread.  The token
  // count is read once per CTA, so every thread works from the same value
  // even if a misordered launch changes it meanwhile.
  // programmatic dependent launch: the next layer's CTAs may take the SM
  // slots this grid frees; this grid's own reads of anything the previous
  // kernel writes come after its wait (mode 1: now; mode 2: once the first
  // stage is in flight)
  if (p.pdl) {
    grid_dep_launch();
    if (p.pdl == 1) grid_dep_wait();
  }
  __shared__ int t_shared[2];
  if (tid == 0) {
    t_shared[0] = __ldcg(p.tokens);
    t_shared[1] = __ldcg(p.nq);
  }
  __syncthreads();
  const int T = t_shared[0];
  if (T <= 0) return;
  const int nq = t_shared[1];             // tokens in key groups (a multiple of G)
  const int r = T - nq;                   // tokens in the FP16 window (at most R)
  const int NS = p.G / kSlice;            // slices per key group (1, 2 or 4)
  const int lgNS = NS == 4 ? 2 : NS - 1;
  const int NR = W >> lgNS;               // key-group records per stage
  const int NGR = nq / p.G;               // key groups per unit
  const int NQS = (NGR + NR - 1) / NR;    // quantized stages per unit
  constexpr uint32_t cq = kCq;                                          // bytes per slice
  constexpr uint32_t cr = kResTile * 4 * D;                             // residual tile bytes
  constexpr int TPS = (SB / cr < static_cast<uint32_t>(W)) ? static_cast<int>(SB / cr) : W;  // tiles per stage
  const int NRT = (r + kResTile - 1) / kResTile;
  const int NRS = (NRT + TPS - 1) / TPS;  // window stages per unit
  const int NI = NQS + NRS;               // stages per unit
  constexpr uint32_t cst_q = W * cq, cst_r = TPS * cr;                  // cost of a stage
  // per-unit setup cost (query tables, warp merge, partial write): measured
  // at about the time a CTA needs for 2*W slices
  constexpr uint32_t csu = 2 * W * (cq > 2048u ? cq : 2048u);
  const uint32_t Cu = csu + static_cast<uint32_t>(NQS) * cst_q + static_cast<uint32_t>(NRS) * cst_r;
  const uint32_t C = static_cast<uint32_t>(p.units) * Cu;
  // a CTA range must hold at least one stage start: range >= largest stage + setup
  const uint32_t maxc = csu + ((NRS > 0 && cst_r > cst_q) || NQS == 0 ? cst_r : cst_q);
  uint32_t peff_u = C / maxc;
  if (peff_u < 1) peff_u = 1;
  if (peff_u > static_cast<uint32_t>(p.grid)) peff_u = p.grid;
  const int pid = blockIdx.x;
  if (pid >= static_cast<int>(peff_u)) return;
  const uint32_t CQ = C / peff_u, CR = C - CQ * peff_u;
  auto range_start = [&](uint32_t pp) -> uint32_t { return pp * CQ + (pp < CR ? pp : CR); };
  // start of stage i of unit u in the cost order
  auto item_start = [&](int u, int i) -> uint32_t {
    return static_cast<uint32_t>(u) * Cu + csu +
           (i < NQS ? static_cast<uint32_t>(i) * cst_q
                    : static_cast<uint32_t>(NQS) * cst_q + static_cast<uint32_t>(i - NQS) * cst_r);
  };
  // first stage starting at or after x, as (unit, stage) with stage < NI
  auto first_item_at = [&](uint32_t x, int& u_out, int& i_out) {
    const uint32_t u = x / Cu;
    const uint32_t ox = x - u * Cu;
    int i;
    if (ox <= csu) {
      i = 0;
    } else {
      const uint32_t o = ox - csu;
      if (NQS > 0 && o <= static_cast<uint32_t>(NQS - 1) * cst_q) i = static_cast<int>((o + cst_q - 1) / cst_q);
      else if (o <= static_cast<uint32_t>(NQS) * cst_q) i = NQS;
      else i = NQS + static_cast<int>((o - static_cast<uint32_t>(NQS) * cst_q + cst_r - 1) / cst_r);
    }
    u_out = static_cast<int>(u);
    i_out = i;
    if (i_out >= NI) {
      ++u_out;
      i_out = 0;
    }
  };
  auto owner_of = [&](uint32_t x) -> int {  // CTA whose range holds cost offset x
    const uint32_t big = CR * (CQ + 1);
    return x < big ? static_cast<int>(x / (CQ + 1)) : static_cast<int>(CR + (x - big) / CQ);
  };
  int u0, i0, u1, i1;
  first_item_at(range_start(pid), u0, i0);
  first_item_at(range_start(pid + 1), u1, i1);
  // flat stage indices f = u*NI + i stay below 2^31: every stage costs more
  // than 1024 of the fewer than 2^32 cost units
  const int f0 = u0 * NI + i0, f1 = u1 * NI + i1;
  const int nst = f1 - f0;                // stages of this CTA
  const int u_first = u0, u_last = i1 == 0 ? u1 - 1 : u1;

  // ---------------- query rows of a unit, double-buffered bulk copies
  // (rows past gqa are never read, the tables test h < gqa)
  uint64_t* full = bars;                  // [kStages] a stage's fill has landed
  uint64_t* qbar = bars + kStages;
  const uint32_t qbytes = static_cast<uint32_t>(p.gqa * D * 2);
  auto issue_q = [&](int u, int buf) {
    mbar_arrive_expect_tx(&qbar[buf], qbytes);
    bulk_g2s(qs + buf * H * D, p.q + static_cast<int64_t>(u) * p.gqa * D, qbytes, &qbar[buf]);
  };
  auto issue_first_q = [&]() {
    issue_q(u_first, 0);
    if (u_first + 1 <= u_last) issue_q(u_first + 1, 1);
  };

  // ---------------- stages: the CTA's k-th stage goes to buffer k % kStages.
  // One thread fills a buffer: the first fills at the start, later ones by
  // the last warp to finish with the buffer's previous fill.  A key-group
  // stage is one bulk copy of NR consecutive records of a unit; a window
  // stage is two copies (keys, values) per 16-token tile.
  auto issue_stage = [&](int k) {
    const int f = f0 + k;
    const int s = k % kStages;
    const int u = f / NI, i = f - u * NI;  // once per stage, one thread
    uint8_t* dst = smem + s * SB;
    if (i < NQS) {
      const int g0 = i * NR;
      const int ng = (NGR - g0 < NR) ? NGR - g0 : NR;
      const uint8_t* src = p.records + u * p.unit_rec_stride + static_cast<int64_t>(g0) * p.rec_bytes;
      const uint32_t bytes = static_cast<uint32_t>(ng * p.rec_bytes);
      // (debug builds: a source outside the cache buffer is recorded and
      // skipped; the stage's barrier still completes)
      if (!in_range(src, bytes, p.buf_lo, p.buf_hi, p.err)) {
        mbar_arrive(&full[s]);
        return;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
      bulk_g2s(dst, src, bytes, &full[s]);
    } else {
      const int t0 = (i - NQS) * TPS;
      const int ntl = (NRT - t0 < TPS) ? NRT - t0 : TPS;
      constexpr uint32_t half = kResTile * D * 2;
      bool ok = true;
      for (int j = 0; j < ntl; ++j) {
        const int slot0 = (nq + (t0 + j) * kResTile) % p.R;
        ok = ok && in_range(p.res_k + u * p.res_stride + static_cast<int64_t>(slot0) * D, half, p.buf_lo, p.buf_hi, p.err) &&
             in_range(p.res_v + u * p.res_stride + static_cast<int64_t>(slot0) * D, half, p.buf_lo, p.buf_hi, p.err);
      }
      if (!ok) {
        mbar_arrive(&full[s]);
        return;
      }
      mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(ntl) * cr);
      for (int j = 0; j < ntl; ++j) {
        const int slot0 = (nq + (t0 + j) * kResTile) % p.R;
        bulk_g2s(dst + j * cr, p.res_k + u * p.res_stride + static_cast<int64_t>(slot0) * D, half, &full[s]);
        bulk_g2s(dst + j * cr + half, p.res_v + u * p.res_stride + static_cast<int64_t>(slot0) * D, half, &full[s]);
      }
    }
  };
  // A warp done reading stage k (every value it read consumed by an
  // instruction) counts itself; the W-th warp of the fill refills the buffer
  // with stage k + kStages.  The counter of a buffer runs over all its fills.
  auto release_stage = [&](int k) {
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      const int s = k % kStages;
      const int prev = atomicAdd(&scnt[s], 1);
      if (prev == (k / kStages + 1) * W - 1 && k + kStages < nst) {
        __threadfence_block();
        fence_proxy_async_smem();  // the warps' reads of the buffer before the copy's writes
        issue_stage(k + kStages);
      }
    }
  };
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      scnt[s] = 0;
    }
    mbar_init(&qbar[0], 1);
    mbar_init(&qbar[1], 1);
    fence_mbar_init();
    // (mode 2: the first stage before the wait, so that the query copy
    // issued after it does not queue behind every stage of every CTA)
    if (p.pdl != 2) {
      issue_first_q();
      for (int k = 0; k < kStages && k < nst; ++k) issue_stage(k);
    } else {
      if (nst > 0) issue_stage(0);
      grid_dep_wait();
      issue_first_q();
      for (int k = 1; k < kStages && k < nst; ++k) issue_stage(k);
    }
  }
  if (p.pdl == 2) {
    // the query, the partials, the split counters and the output may belong
    // to the previous kernel's work: everything after this waits for it
    grid_dep_wait();
  }
  __syncthreads();  // barriers initialised before anyone waits on them

  const __half2 negmask = part ? __float2half2_rn(-1.0f) : __float2half2_rn(0.0f);
  const float alpha = p.alpha;  // residual scores (fp16 keys)
  // quantized scores carry 2^(Pmax - 24) (subnormal codes, scaled query)
  const float alpha_q = p.alpha * (16777216.0f / static_cast<float>(1 << key_pos_max<KB>()));
  const uint32_t vhalf_sel = (g & 1) ? 0x7632u : 0x5410u;  // 2-bit values, D = 64
  bool failed = false;
  const int team = warp >> lgNS, sl = warp & (NS - 1);  // record of a stage and 32-token slice of it
  int k = 0;        // the CTA's stage
  int si = i0;      // its index in the unit

  for (int u = u_first; u <= u_last; ++u) {
    const int i_end = (u == u1) ? i1 : NI;
    const int b = u / p.kv_heads, kvh = u - b * p.kv_heads;

    // ---------------- per-unit query tables (from the prefetched query rows)
    const int seg = u - u_first;
    const __half* qu = qs + (seg & 1) * H * D;
    if (!failed && !mbar_wait(&qbar[seg & 1], static_cast<uint32_t>((seg >> 1) & 1), p.err)) failed = true;
    if constexpr (kT) {
      // lane (g, tig): head g, channel pairs key_pair_channels(tig, pi)
      const int h = g;
      const bool live = h < p.gqa;
      // (each head's lanes start at another pair: the eight query rows are
      // D/2 words apart, so the same pair of all heads would share a bank)
      for (int pr = warp; pr < NPK; pr += W) {
        const int pi = (pr + 2 * g) % NPK;
        int ca, cb;
        key_pair_channels<KB, D>(tig, pi, ca, cb);
        const __half z0 = __float2half(0.0f);
        const __half2 q2 = __halves2half2(live ? qu[h * D + ca] : z0, live ? qu[h * D + cb] : z0);
        qp_tab[kt_idx(0, pi, lane)] = h2_as_u32(q2);
        const float f = static_cast<float>(1 << (key_pos_max<KB>() - key_pos<KB, D>(pi)));
        qps_tab[kt_idx(0, pi, lane)] = h2_as_u32(__hmul2(q2, __float2half2_rn(f)));
      }
      // window keys (natural channel order): channels 16kk + 8rr + 2tig, +1
      for (int kr = warp; kr < KS; kr += W) {
        const int kk = (kr + g) % KS;
        for (int rr = 0; rr < 2; ++rr) {
          const int c = 16 * kk + 8 * rr + 2 * tig;
          qr_tab[rt_idx(0, kk, lane) + rr] = live ? h2_as_u32(__halves2half2(qu[h * D + c], qu[h * D + c + 1])) : 0u;
        }
      }
      if constexpr (KM == 1) {
        constexpr float kSS = static_cast<float>(1 << key_pos_max<KB>()) / 16777216.0f;
        for (int hh = warp; hh < H; hh += W) {
          float sum = 0.0f;
#pragma unroll
          for (int c = lane; c < D; c += 32) sum += __half2float(qu[hh * D + c]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          if (lane == 0) qsum_s[hh] = hh < p.gqa ? sum * kSS : 0.0f;
        }
      }
    } else {
      // every warp fills a quarter of the per-lane tables (lane = tid & 31)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int h = 4 * j + (g >> 1);
        const bool live = h < p.gqa;
        for (int pr = warp; pr < NPK; pr += W) {
          const int pi = (pr + 2 * (g >> 1)) % NPK;  // (bank spread, as above)
          int ca, cb;
          key_pair_channels<KB, D>(tig, pi, ca, cb);
          const __half z0 = __float2half(0.0f);
          const __half qa = (live && ca >= 0) ? qu[h * D + ca] : z0;
          const __half qb = (live && cb >= 0) ? qu[h * D + cb] : z0;
          const __half2 q2 = __halves2half2(qa, qb);
          qp_tab[kt_idx(j, pi, lane)] = h2_as_u32(q2);
          const float f = static_cast<float>(1 << (key_pos_max<KB>() - key_pos<KB, D>(pi)));
          const uint32_t scaled = h2_as_u32(__hmul2(q2, __float2half2_rn(f)));
          // per-token keys: the scaled query is the whole B operand (hi column; lo = 0)
          qps_tab[kt_idx(j, pi, lane)] = (KM == 1 && part) ? 0u : scaled;
        }
        for (int kr = warp; kr < KS; kr += W) {
          const int kk = (kr + (g >> 1)) % KS;
          for (int rr = 0; rr < 2; ++rr) {
            const int c = 16 * kk + 8 * rr + 2 * tig;
            qr_tab[rt_idx(j, kk, lane) + rr] =
                (live && !part) ? h2_as_u32(__halves2half2(qu[h * D + c], qu[h * D + c + 1])) : 0u;
          }
        }
      }
      if constexpr (KM == 1) {
        // per head: sum_c q_c (scaled like the scores), for the keys' zero term
        constexpr float kSS = static_cast<float>(1 << key_pos_max<KB>()) / 16777216.0f;
        for (int h = warp; h < H; h += W) {
          float sum = 0.0f;
#pragma unroll
          for (int c = lane; c < D; c += 32) sum += __half2float(qu[h * D + c]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          if (lane == 0) qsum_s[h] = h < p.gqa ? sum * kSS : 0.0f;
        }
      }
    }
    __syncthreads();
    if (tid == 0 && u + 2 <= u_last) issue_q(u + 2, seg & 1);
    // per-token keys: the B operand of the scores is fixed for the unit
    uint32_t bqu[KM == 1 ? NT : 1][KM == 1 ? NPK : 1];
    float qsj[NT];
    if constexpr (KM == 1 && kT) {
      qsj[0] = qsum_s[g];
#pragma unroll
      for (int pi = 0; pi < NPK; pi += 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(qps_tab + kt_idx(0, pi, lane));
        bqu[0][pi] = v.x;
        bqu[0][pi + 1] = v.y;
      }
    } else if constexpr (KM == 1) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        qsj[j] = qsum_s[4 * j + tig];
#pragma unroll
        for (int pi = 0; pi < NPK; pi += 2) {
          const uint2 v = *reinterpret_cast<const uint2*>(qps_tab + kt_idx(j, pi, lane));
          bqu[j][pi] = v.x;
          bqu[j][pi + 1] = v.y;
        }
      }
    }

    // ---------------- warp state for this unit
    float m[NT], l[NT], vb[NT];
    float acc[MTA][NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.0f;
      vb[j] = 0.0f;
#pragma unroll
      for (int mt = 0; mt < MTA; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.0f;
    }
    bool has_q = false, in_res = false, dumped = false;
    // transposed form: this lane's head g; rows g (hi) and g + 8 (lo) of the
    // P.V accumulator, n-tile c = 8 channels
    float m1 = -INFINITY, l1 = 0.0f, vb1 = 0.0f;
    float acc2[kT ? NEV : 1][4];
#pragma unroll
    for (int c = 0; c < (kT ? NEV : 1); ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2[c][e] = 0.0f;
    // online-softmax update of the transposed form: tmax = this lane's maximum
    auto softmax_update1 = [&](float tmax_in) {
      if (__any_sync(0xffffffffu, tmax_in > m1 + 8.0f)) {
        float t = fmaxf(tmax_in, __shfl_xor_sync(0xffffffffu, tmax_in, 1));
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 2));
        const float mn = fmaxf(m1, t);
        const float f = (mn == -INFINITY) ? 1.0f : ex2(m1 - mn);
        m1 = mn;
        l1 *= f;
        vb1 *= f;
#pragma unroll
        for (int c = 0; c < (kT ? NEV : 1); ++c)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[c][e] *= f;
      }
    };
    // the key group whose scaled-query table this warp holds (per-channel keys)
    int tab_g = -1;
    float bias_g[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) bias_g[j] = 0.0f;

    // online-softmax update: tmax = max of this tile's scaled scores per head
    auto softmax_update = [&](const float (&tmax_in)[NT]) {
      // m only moves when some lane's own maximum passes it by more than 8
      // (log2 units); the lanes of a head reduce their maxima only then
      bool need = false;
#pragma unroll
      for (int j = 0; j < NT; ++j) need |= tmax_in[j] > m[j] + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float t = tmax_in[j];
          t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 4));
          t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 8));
          t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 16));
          const float mn = fmaxf(m[j], t);
          const float f = (mn == -INFINITY) ? 1.0f : ex2(m[j] - mn);
          m[j] = mn;
          l[j] *= f;
          vb[j] *= f;
#pragma unroll
          for (int mt = 0; mt < MTA; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][j][e] *= f;
        }
      }
    };

    // PV B fragments from (p~ of rows g, g+8) pairs: the thread's column is
    // (head 4j + g/2, hi or lo); tokens come from lanes srcA and srcA + dB
    auto pv_b = [&](uint32_t hi, uint32_t lo, int srcA, int dB, uint32_t& b01, uint32_t& b23) {
      const uint32_t xh = __shfl_sync(0xffffffffu, hi, srcA);
      const uint32_t yh = __shfl_sync(0xffffffffu, hi, srcA + dB);
      const uint32_t xl = __shfl_sync(0xffffffffu, lo, srcA);
      const uint32_t yl = __shfl_sync(0xffffffffu, lo, srcA + dB);
      const uint32_t x = part ? xl : xh, y = part ? yl : yh;
      b01 = prmt(x, y, 0x5410u);
      b23 = prmt(x, y, 0x7632u);
    };

    for (; si < i_end; ++si, ++k) {
      const int i = si;
      if (!failed && !mbar_wait(&full[k % kStages], static_cast<uint32_t>((k / kStages) & 1), p.err)) failed = true;
      const uint8_t* stg = smem + (k % kStages) * SB;
      // this warp's share of the stage: slice sl of record `team`, or window tile `warp`
      const bool q_item = i < NQS && i * NR + team < NGR;
      const int tile = (i - NQS) * TPS + warp;
      const bool r_item = i >= NQS && warp < TPS && tile < NRT;
      // Counts the warp done with the stage (refilling it if last).  Every
      // value read from the stage must have been consumed by an instruction first.
      bool released = false;
      auto release_slot = [&]() {
        release_stage(k);
        released = true;
      };

      if (failed) {
        // a copy never landed: skip the work, keep the control flow
      } else if (kT && q_item) {
        // ============ quantized slice, transposed form (8 heads x {hi, lo} rows)
        has_q = true;
        const uint32_t* rec = reinterpret_cast<const uint32_t*>(stg + team * p.rec_bytes);
        const int t0 = sl * kSlice;
        const uint32_t* Kc = rec + t0 * WK;
        const uint32_t* Vc = rec + p.G * WK + t0 * WV;
        const __half* Ks = reinterpret_cast<const __half*>(rec + p.G * (WK + WV));
        const __half* Kz = Ks + D;
        const __half2* Ksz = reinterpret_cast<const __half2*>(rec + p.G * (WK + WV)) + t0;
        const __half2* Vsz = (KM == 0 ? reinterpret_cast<const __half2*>(Kz + D) : Ksz - t0 + p.G) + t0;
        constexpr float kScoreScale = static_cast<float>(1 << key_pos_max<KB>()) / 16777216.0f;
        constexpr int WT = KS_::WT, PW = KS_::PW;
        // per-channel keys: the group's key scale (pairs, for q~ = q s) and the
        // zero term sum_c q_c z_c of head g (one MMA chain, q in row g)
        uint32_t sp[KM == 0 ? NPK : 1];
        float bias1 = 0.0f;
        if constexpr (KM == 0) {
          uint32_t zp[NPK];
          uint32_t zn[NPK], sn[NPK];
          // chunk j of this lane's channel quarter tig is stored chunk 4j + tig
          const uint4* zsrc = reinterpret_cast<const uint4*>(Kz) + tig;
          const uint4* ssrc = reinterpret_cast<const uint4*>(Ks) + tig;
#pragma unroll
          for (int pi = 0; pi < NPK; pi += 4) {
            const uint4 vz = zsrc[pi];
            const uint4 vs = ssrc[pi];
            zn[pi] = vz.x; zn[pi + 1] = vz.y; zn[pi + 2] = vz.z; zn[pi + 3] = vz.w;
            sn[pi] = vs.x; sn[pi + 1] = vs.y; sn[pi + 2] = vs.z; sn[pi + 3] = vs.w;
          }
#pragma unroll
          for (int wi = 0; wi < WT; ++wi) {
            const uint32_t* nz = zn + wi * PW;
            const uint32_t* ns = sn + wi * PW;
            uint32_t* oz = zp + wi * PW;
            uint32_t* os = sp + wi * PW;
            if constexpr (KB == 4) {
              oz[0] = prmt(nz[0], nz[2], 0x5410u); oz[1] = prmt(nz[0], nz[2], 0x7632u);
              oz[2] = prmt(nz[1], nz[3], 0x5410u); oz[3] = prmt(nz[1], nz[3], 0x7632u);
              os[0] = prmt(ns[0], ns[2], 0x5410u); os[1] = prmt(ns[0], ns[2], 0x7632u);
              os[2] = prmt(ns[1], ns[3], 0x5410u); os[3] = prmt(ns[1], ns[3], 0x7632u);
            } else if constexpr (KB == 2) {
#pragma unroll
              for (int kq = 0; kq < 4; ++kq) {
                oz[2 * kq] = prmt(nz[kq], nz[kq + 4], 0x5410u);
                oz[2 * kq + 1] = prmt(nz[kq], nz[kq + 4], 0x7632u);
                os[2 * kq] = prmt(ns[kq], ns[kq + 4], 0x5410u);
                os[2 * kq + 1] = prmt(ns[kq], ns[kq + 4], 0x7632u);
              }
            } else {
              oz[0] = prmt(nz[0], nz[1], 0x5410u); oz[1] = prmt(nz[0], nz[1], 0x7632u);
              os[0] = prmt(ns[0], ns[1], 0x5410u); os[1] = prmt(ns[0], ns[1], 0x7632u);
            }
          }
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < KSK; ++kk) {
            const uint2 qv = *reinterpret_cast<const uint2*>(qp_tab + kt_idx(0, 2 * kk, lane));
            mma_16816((kk & 1) ? c1 : c0, qv.x, 0u, qv.y, 0u, zp[2 * kk], zp[2 * kk + 1]);
          }
          bias1 = (c0[0] + c1[0]) * kScoreScale;  // row g: head g, in the scaled score domain
        }
        // ---- scores of the slice's 32 tokens: n-tile n = tokens 8n..8n+7,
        // column 2tig + e = token 8n + 2tig + e; rows g (hi part) and g + 8 (lo)
        // one accumulator chain per n-tile, started at the key zero term (row g)
        float sc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[n][e] = (e < 2) ? bias1 : 0.0f;
        {
          uint32_t wr[4][WT];
#pragma unroll
          for (int rw = 0; rw < 4; ++rw)
            lds_row_words<WT>(wr[rw], Kc + (8 * rw + g) * WK, tig * WT, code_word_xor(WK, true, g));
#pragma unroll
          for (int wi = 0; wi < WT; ++wi) {
            uint32_t e[4][PW];
#pragma unroll
            for (int rw = 0; rw < 4; ++rw) k_word_pairs<KB>(wr[rw][wi], e[rw]);
#pragma unroll
            for (int k2 = 0; k2 < PW / 2; ++k2) {
              const int kk = wi * (PW / 2) + k2;
              // A of k-step kk: q~ = q s of head g as fp16 hi (row g) + lo (row g + 8)
              uint32_t a0, a1, a2, a3;
              if constexpr (KM == 0) {
                const uint2 q2 = *reinterpret_cast<const uint2*>(qps_tab + kt_idx(0, 2 * kk, lane));
                const __half2 qa = u32_as_h2(q2.x), qb = u32_as_h2(q2.y);
                const __half2 sa = u32_as_h2(sp[2 * kk]), sb = u32_as_h2(sp[2 * kk + 1]);
                const __half2 ha = __hmul2(qa, sa), hb = __hmul2(qb, sb);
                a0 = h2_as_u32(ha);
                a1 = h2_as_u32(__hfma2(qa, sa, __hneg2(ha)));
                a2 = h2_as_u32(hb);
                a3 = h2_as_u32(__hfma2(qb, sb, __hneg2(hb)));
              } else {
                a0 = bqu[0][2 * kk];
                a1 = 0u;
                a2 = bqu[0][2 * kk + 1];
                a3 = 0u;
              }
#pragma unroll
              for (int n = 0; n < 4; ++n)
                mma_16816(sc[n], a0, a1, a2, a3, e[n][2 * k2], e[n][2 * k2 + 1]);
            }
          }
        }
        // ---- value code words (tokens 16kb + 2tig, +1, +8, +9), the tokens'
        // value (scale, zero) and per-token key (scale, zero): the last reads
        constexpr int VW = VS_::VW;
        const int voff = (VB == 2 && D == 64) ? (g >> 1) : g * VW;
        // (lanes with tig >= 2 read the odd token of each pair first: rows
        // 0, 2, 5, 7, then 1, 3, 4, 6 of a pair group hit four different
        // quarters of the banks for 32-byte rows)
        uint32_t vw[2][4][VW];
        const int sw = tig >> 1;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int pr = 0; pr < 2; ++pr) {
            const int ra = 16 * kb + 8 * pr + 2 * tig + sw, rb = 16 * kb + 8 * pr + 2 * tig + 1 - sw;
            uint32_t wa[VW], wb[VW];
            lds_row_words<VW>(wa, Vc + ra * WV, voff, code_word_xor(WV, false, ra));
            lds_row_words<VW>(wb, Vc + rb * WV, voff, code_word_xor(WV, false, rb));
#pragma unroll
            for (int x = 0; x < VW; ++x) {
              vw[kb][2 * pr][x] = sw ? wb[x] : wa[x];
              vw[kb][2 * pr + 1][x] = sw ? wa[x] : wb[x];
            }
          }
        float2 vsz[4][2], ksz[KM == 1 ? 4 : 1][2];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const uint2 v2 = *reinterpret_cast<const uint2*>(Vsz + 8 * n + 2 * tig);
          vsz[n][0] = __half22float2(u32_as_h2(v2.x));
          vsz[n][1] = __half22float2(u32_as_h2(v2.y));
          if constexpr (KM == 1) {
            const uint2 k2 = *reinterpret_cast<const uint2*>(Ksz + 8 * n + 2 * tig);
            ksz[n][0] = __half22float2(u32_as_h2(k2.x));
            ksz[n][1] = __half22float2(u32_as_h2(k2.y));
          }
        }
        release_slot();

        // ---- softmax over head g's 8 tokens of this lane
        float sv[4][2];
        float tmax = -INFINITY;
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if constexpr (KM == 1) {
              sv[n][e] = fmaf(ksz[n][e].x, sc[n][e], ksz[n][e].y * qsj[0]);
            } else {
              sv[n][e] = sc[n][e] + sc[n][e + 2];
            }
            tmax = fmaxf(tmax, sv[n][e]);
          }
        softmax_update1(alpha_q * tmax);
        uint32_t ph[4], pl[4];  // P~ = p s_v of tokens (8n + 2tig, +1) as fp16 hi + lo
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const float pa = ex2(fmaf(sv[n][0], alpha_q, -m1)), pb = ex2(fmaf(sv[n][1], alpha_q, -m1));
          l1 += pa + pb;
          vb1 = fmaf(pa, vsz[n][0].y, fmaf(pb, vsz[n][1].y, vb1));
          split_pair(pa * vsz[n][0].x, pb * vsz[n][1].x, ph[n], pl[n]);
        }
        // ---- P~.V: k-block kb = tokens 16kb..16kb+15 (n-tiles 2kb, 2kb + 1)
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          uint32_t hvt[2][NEV];
          v_pairs<VB, D>(vw[kb][0], vw[kb][1], vhalf_sel, hvt[0]);
          v_pairs<VB, D>(vw[kb][2], vw[kb][3], vhalf_sel, hvt[1]);
#pragma unroll
          for (int c = 0; c < NEV; ++c)
            mma_16816(acc2[c], ph[2 * kb], pl[2 * kb], ph[2 * kb + 1], pl[2 * kb + 1], hvt[0][c], hvt[1][c]);
        }
      } else if (!kT && q_item) {
        // ============ quantized slice of a key group (32 tokens)
        has_q = true;
        // the record's layout: [K rows G x WK][V rows G x WV][key (scale, zero)][V (scale, zero) G pairs]
        const uint32_t* rec = reinterpret_cast<const uint32_t*>(stg + team * p.rec_bytes);
        const int t0 = sl * kSlice;
        const uint32_t* Kc = rec + t0 * WK;
        const uint32_t* Vc = rec + p.G * WK + t0 * WV;
        const __half* Ks = reinterpret_cast<const __half*>(rec + p.G * (WK + WV));  // per-channel keys
        const __half* Kz = Ks + D;
        const __half2* Ksz = reinterpret_cast<const __half2*>(rec + p.G * (WK + WV)) + t0;  // per-token keys
        const __half2* Vsz = (KM == 0 ? reinterpret_cast<const __half2*>(Kz + D) : Ksz - t0 + p.G) + t0;
        float bias[NT];
        uint32_t bq[NT][kTabSmem ? 1 : NPK];
        if constexpr (KM == 1) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            bias[j] = 0.0f;
#pragma unroll
            for (int pi = 0; pi < NPK; ++pi) bq[j][pi] = bqu[j][pi];
          }
        } else {
        const int grp = i * NR + team;
        if (!kTabSmem || grp != tab_g) {
        tab_g = grp;
        uint32_t qp[NT][NPK];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int pi = 0; pi < NPK; pi += 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(qp_tab + kt_idx(j, pi, lane));
            qp[j][pi] = v.x;
            qp[j][pi + 1] = v.y;
          }
        // key codes arrive as code * 2^(pos - 24): the scaled query carries
        // 2^(Pmax - pos), so every score product is scaled by 2^(Pmax - 24)
        constexpr float kScoreScale = static_cast<float>(1 << key_pos_max<KB>()) / 16777216.0f;
        // zero and scale pairs in key-pair order
        uint32_t zp[NPK], sp[NPK];
        if constexpr (KB == 3) {
#pragma unroll
          for (int pi = 0; pi < NPK; ++pi) {
            int ca, cb;
            key_pair_channels<KB, D>(tig, pi, ca, cb);
            const __half h0 = __float2half(0.0f);
            zp[pi] = h2_as_u32(__halves2half2(ca >= 0 ? Kz[ca] : h0, cb >= 0 ? Kz[cb] : h0));
            sp[pi] = h2_as_u32(__halves2half2(ca >= 0 ? Ks[ca] : h0, cb >= 0 ? Ks[cb] : h0));
          }
        } else {
          constexpr int PW = KS_::PW;
          uint32_t zn[NPK], sn[NPK];
          // chunk j of this lane's channel quarter tig is stored chunk 4j + tig
          const uint4* zsrc = reinterpret_cast<const uint4*>(Kz) + tig;
          const uint4* ssrc = reinterpret_cast<const uint4*>(Ks) + tig;
#pragma unroll
          for (int pi = 0; pi < NPK; pi += 4) {
            const uint4 vz = zsrc[pi];
            const uint4 vs = ssrc[pi];
            zn[pi] = vz.x; zn[pi + 1] = vz.y; zn[pi + 2] = vz.z; zn[pi + 3] = vz.w;
            sn[pi] = vs.x; sn[pi + 1] = vs.y; sn[pi + 2] = vs.z; sn[pi + 3] = vs.w;
          }
#pragma unroll
          for (int wi = 0; wi < KS_::WT; ++wi) {
            const uint32_t* nz = zn + wi * PW;
            const uint32_t* ns = sn + wi * PW;
            uint32_t* oz = zp + wi * PW;
            uint32_t* os = sp + wi * PW;
            if constexpr (KB == 4) {
              oz[0] = prmt(nz[0], nz[2], 0x5410u); oz[1] = prmt(nz[0], nz[2], 0x7632u);
              oz[2] = prmt(nz[1], nz[3], 0x5410u); oz[3] = prmt(nz[1], nz[3], 0x7632u);
              os[0] = prmt(ns[0], ns[2], 0x5410u); os[1] = prmt(ns[0], ns[2], 0x7632u);
              os[2] = prmt(ns[1], ns[3], 0x5410u); os[3] = prmt(ns[1], ns[3], 0x7632u);
            } else if constexpr (KB == 2) {
#pragma unroll
              for (int kq = 0; kq < 4; ++kq) {
                oz[2 * kq] = prmt(nz[kq], nz[kq + 4], 0x5410u);
                oz[2 * kq + 1] = prmt(nz[kq], nz[kq + 4], 0x7632u);
                os[2 * kq] = prmt(ns[kq], ns[kq + 4], 0x5410u);
                os[2 * kq + 1] = prmt(ns[kq], ns[kq + 4], 0x7632u);
              }
            } else {
              oz[0] = prmt(nz[0], nz[1], 0x5410u); oz[1] = prmt(nz[0], nz[1], 0x7632u);
              os[0] = prmt(ns[0], ns[1], 0x5410u); os[1] = prmt(ns[0], ns[1], 0x7632u);
            }
          }
        }
        // bias = sum_c q_c z_c: MMAs with the zeros broadcast over rows (two chains)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < KSK; ++kk)
            mma_16816((kk & 1) ? c1 : c0, zp[2 * kk], zp[2 * kk], zp[2 * kk + 1], zp[2 * kk + 1], qp[j][2 * kk],
                      qp[j][2 * kk + 1]);
          bias_g[j] = (c0[0] + c1[0]) * kScoreScale;  // in the scaled score domain
        }
        // folded query q~ = q * s (scaled): hi part in even columns, lo part in odd ones
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int pi = 0; pi < NPK; pi += 2) {
            const uint2 q2 = *reinterpret_cast<const uint2*>(qps_tab + kt_idx(j, pi, lane));
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t qsc = h2 ? q2.y : q2.x;
              const int pj = pi + h2;
              if constexpr (KB == 3) {
                // fp32 products: the 2-bit fields use s2 = (s*7)/3 (an fp32 value)
                int ca, cb;
                key_pair_channels<KB, D>(tig, pj, ca, cb);
                const float2 qf = __half22float2(u32_as_h2(qsc));
                float2 sf = __half22float2(u32_as_h2(sp[pj]));
                if (ca >= 0 && ca % 11 == 10) sf.x = __fdiv_rn(__fmul_rn(sf.x, 7.0f), 3.0f);
                if (cb >= 0 && cb % 11 == 10) sf.y = __fdiv_rn(__fmul_rn(sf.y, 7.0f), 3.0f);
                uint32_t hi, lo;
                split_pair(qf.x * sf.x, qf.y * sf.y, hi, lo);
                bq[j][kTabSmem ? 0 : pj] = part ? lo : hi;
              } else {
                const __half2 qq = u32_as_h2(qsc);
                const __half2 ss = u32_as_h2(sp[pj]);
                const __half2 hi = __hmul2(qq, ss);
                const uint32_t v = h2_as_u32(__hfma2(qq, ss, __hmul2(hi, negmask)));
                if constexpr (kTabSmem) qtab[kt_idx(j, pj, lane)] = v;
                else bq[j][pj] = v;
              }
            }
          }
        if constexpr (kTabSmem) __syncwarp();
        }  // table of the group
#pragma unroll
        for (int j = 0; j < NT; ++j) bias[j] = bias_g[j];
        }  // per-channel keys

        // ---- scores of the slice's 32 tokens: tiles 0 (tokens 0..15) and 1 (16..31);
        // rows g and g+8 of each; two accumulator chains per tile (the bias is
        // added afterwards, so these chains do not wait for the bias MMAs)
        float sc[2][NT][4];
        {
          float sx[2][NT][4];
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                sc[t][j][q4] = 0.0f;
                sx[t][j][q4] = 0.0f;
              }
          // B operand of k-step kk for head tile j
          auto bq_at = [&](int j, int kk, uint32_t& b0, uint32_t& b1) {
            if constexpr (kTabSmem && KM == 0) {
              const uint2 v = *reinterpret_cast<const uint2*>(qtab + kt_idx(j, 2 * kk, lane));
              b0 = v.x;
              b1 = v.y;
            } else {
              b0 = bq[j][2 * kk];
              b1 = bq[j][2 * kk + 1];
            }
          };
          if constexpr (KB == 3) {
            uint32_t e[4][NPK];
#pragma unroll
            for (int rw = 0; rw < 4; ++rw) key_row_pairs<KB, D>(Kc + (8 * rw + g) * WK, tig, e[rw]);
#pragma unroll
            for (int kk = 0; kk < KSK; ++kk)
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                uint32_t b0, b1;
                bq_at(j, kk, b0, b1);
#pragma unroll
                for (int t = 0; t < 2; ++t)
                  mma_16816((kk & 1) ? sx[t][j] : sc[t][j], e[2 * t][2 * kk], e[2 * t + 1][2 * kk],
                            e[2 * t][2 * kk + 1], e[2 * t + 1][2 * kk + 1], b0, b1);
              }
          } else {
            // one code word of each of the 4 rows at a time: its PW pairs
            // feed PW/2 k-steps
            constexpr int WT = KS_::WT, PW = KS_::PW;
            uint32_t wr[4][WT];
#pragma unroll
            for (int rw = 0; rw < 4; ++rw)
              lds_row_words<WT>(wr[rw], Kc + (8 * rw + g) * WK, tig * WT, code_word_xor(WK, true, g));
#pragma unroll
            for (int wi = 0; wi < WT; ++wi) {
              uint32_t e[4][PW];
#pragma unroll
              for (int rw = 0; rw < 4; ++rw) k_word_pairs<KB>(wr[rw][wi], e[rw]);
#pragma unroll
              for (int k2 = 0; k2 < PW / 2; ++k2) {
                const int kk = wi * (PW / 2) + k2;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                  uint32_t b0, b1;
                  bq_at(j, kk, b0, b1);
#pragma unroll
                  for (int t = 0; t < 2; ++t)
                    mma_16816((kk & 1) ? sx[t][j] : sc[t][j], e[2 * t][2 * k2], e[2 * t + 1][2 * k2],
                              e[2 * t][2 * k2 + 1], e[2 * t + 1][2 * k2 + 1], b0, b1);
                }
              }
            }
          }
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) sc[t][j][q4] += sx[t][j][q4];
        }

        // ---- value codes of both tiles, read before the slot is released:
        // 3-bit values are unpacked here, the others keep their code words
        // and are unpacked just before their P.V
        constexpr int NE = (VB == 3) ? 2 * VS_::MT3 : NP;
        constexpr int VW = VS_::VW;
        uint32_t hv[VB == 3 ? 2 : 1][2][VB == 3 ? NE : 1];   // [tile][token pair (tig,tig+4) | (tig+8,tig+12)][entry]
        uint32_t h2v[2][2][2];   // 3-bit values: 2-bit-field tile entries
        uint32_t vw[2][4][VW];   // other widths: [tile][token tig + 4r][word]
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int tb = 16 * t;
          if constexpr (VB == 3) {
            uint32_t wa[4], wbw[4];
            const int wA = (D == 128) ? g : (g < 6 ? g : 0);
            const int wB = 8 + (g >> 1);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint32_t* row = Vc + (tb + tig + 4 * q4) * WV;
              wa[q4] = (D == 128 || g < 6) ? row[wA] : 0u;
              wbw[q4] = (D == 128) ? row[wB] : 0u;
            }
            const int hsh = 15 * (g & 1);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
              uint32_t* Hh = hv[t][pr];
              const uint32_t a0 = wa[2 * pr], a1 = wa[2 * pr + 1];
              lo5(a0, a1, Hh);
              lo5(a0 >> 15, a1 >> 15, Hh + 5);
              h2v[t][pr][0] = (D == 128 || g < 5) ? slot10_pair(a0, a1) : 0u;
              if constexpr (D == 128) {
                const uint32_t b0 = wbw[2 * pr], b1 = wbw[2 * pr + 1];
                lo5(b0 >> hsh, b1 >> hsh, Hh + 10);
                Hh[15] = 0u;
                h2v[t][pr][1] = ((g & 1) == 0 && wB <= 10) ? slot10_pair(b0, b1) : 0u;
              } else {
                h2v[t][pr][1] = 0u;
              }
            }
          } else {
            const int voff = (VB == 2 && D == 64) ? (g >> 1) : g * VW;
#pragma unroll
            for (int r4 = 0; r4 < 4; ++r4)
              lds_row_words<VW>(vw[t][r4], Vc + (tb + tig + 4 * r4) * WV, voff, code_word_xor(WV, false, tig));
          }
        }

        // the last reads of the slot: each token's value (scale, zero); after
        // them the slot is free for the next copy while the softmax and P.V run
        float2 sz[2][2], kz2[2][2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          sz[t][0] = __half22float2(Vsz[16 * t + g]);
          sz[t][1] = __half22float2(Vsz[16 * t + g + 8]);
          if constexpr (KM == 1) {
            kz2[t][0] = __half22float2(Ksz[16 * t + g]);
            kz2[t][1] = __half22float2(Ksz[16 * t + g + 8]);
          }
        }
        release_slot();

        // raw scores: s[t][j][0] token 16t+g, [1] token 16t+g+8; m is kept in
        // units of alpha * raw (log2 domain), p = 2^(alpha*raw - m)
        float s[2][NT][2];
        float tmax[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if constexpr (KM == 1) {  // s_t * (q . codes_t) + z_t * sum(q), per token
              s[t][j][0] = fmaf(kz2[t][0].x, sc[t][j][0] + sc[t][j][1], kz2[t][0].y * qsj[j]);
              s[t][j][1] = fmaf(kz2[t][1].x, sc[t][j][2] + sc[t][j][3], kz2[t][1].y * qsj[j]);
            } else {
              s[t][j][0] = (sc[t][j][0] + sc[t][j][1]) + bias[j];
              s[t][j][1] = (sc[t][j][2] + sc[t][j][3]) + bias[j];
            }
          }
          tmax[j] = alpha_q * fmaxf(fmaxf(s[0][j][0], s[0][j][1]), fmaxf(s[1][j][0], s[1][j][1]));
        }
        softmax_update(tmax);
        const int srcA = 4 * tig + (g >> 1);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint32_t b01[NT], b23[NT], c01[NT], c23[NT];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const float pa = ex2(fmaf(s[t][j][0], alpha_q, -m[j])), pb = ex2(fmaf(s[t][j][1], alpha_q, -m[j]));
            l[j] += pa + pb;
            vb[j] = fmaf(pa, sz[t][0].y, fmaf(pb, sz[t][1].y, vb[j]));
            uint32_t hi, lo;
            split_pair(pa * sz[t][0].x, pb * sz[t][1].x, hi, lo);
            pv_b(hi, lo, srcA, 16, b01[j], b23[j]);  // tokens (tig, tig+4 | tig+8, tig+12)
            if constexpr (VB == 3) {
              const float s2a = __fdiv_rn(__fmul_rn(sz[t][0].x, 7.0f), 3.0f);
              const float s2b = __fdiv_rn(__fmul_rn(sz[t][1].x, 7.0f), 3.0f);
              split_pair(pa * s2a, pb * s2b, hi, lo);
              pv_b(hi, lo, srcA, 16, c01[j], c23[j]);
            }
          }
          // ---- p~.V over tokens 16t + (tig, tig+4 | tig+8, tig+12), rows = channels
          if constexpr (VB == 3) {
            constexpr int MT3 = VS_::MT3;
            // rows g / g+8 of tile mt (see vq_channel): d128 pairs entries of equal
            // bit position, d64 takes fields mt / 5 + mt of the same word
            constexpr int lo128[8] = {0, 5, 10, 1, 6, 11, 2, 12}, hi128[8] = {3, 8, 13, 4, 9, 14, 7, 15};
#pragma unroll
            for (int mt = 0; mt < MT3; ++mt) {
              const int el = (D == 128) ? lo128[mt] : mt, eh = (D == 128) ? hi128[mt] : MT3 + mt;
#pragma unroll
              for (int j = 0; j < NT; ++j)
                mma_16816(acc[mt][j], hv[t][0][el], hv[t][0][eh], hv[t][1][el], hv[t][1][eh], b01[j], b23[j]);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j)
              mma_16816(acc[MT3][j], h2v[t][0][0], h2v[t][0][1], h2v[t][1][0], h2v[t][1][1], c01[j], c23[j]);
          } else {
            uint32_t hvt[2][NE];
            v_pairs<VB, D>(vw[t][0], vw[t][1], vhalf_sel, hvt[0]);
            v_pairs<VB, D>(vw[t][2], vw[t][3], vhalf_sel, hvt[1]);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
              for (int j = 0; j < NT; ++j)
                mma_16816(acc[mt][j], hvt[0][mt], hvt[0][KS + mt], hvt[1][mt], hvt[1][KS + mt], b01[j], b23[j]);
          }
        }
      } else if (kT && r_item) {
        // ============ residual tile, transposed form
        if (!in_res) {
          if (has_q) {
            // park the quantized-token part (its channel map: column 2tig + e of
            // n-tile c is channel (2tig + e) * D/8 + c) in wo
            float vbt = vb1 + __shfl_xor_sync(0xffffffffu, vb1, 1);
            vbt += __shfl_xor_sync(0xffffffffu, vbt, 2);
            vb1 = 0.0f;
            float* dd = wo + (warp * H + g) * D;
#pragma unroll
            for (int c = 0; c < NEV; ++c) {
              const float fs = 16777216.0f / static_cast<float>(1 << value_pos<VB, D>(c % KS));
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                dd[wo_chan<true>(g, (2 * tig + e) * (D / 8) + c)] = fmaf(acc2[c][e] + acc2[c][e + 2], fs, vbt);
                acc2[c][e] = 0.0f;
                acc2[c][e + 2] = 0.0f;
              }
            }
            if (tig == 0) dm[warp * H + g] = m1;
            dumped = true;
          }
          in_res = true;
        }
        const __half* Kr = reinterpret_cast<const __half*>(stg + warp * cr);
        const __half* Vr = Kr + kResTile * D;
        const int left = r - tile * kResTile;
        const int vt = left < kResTile ? left : kResTile;
        // scores: rows g = head g (fp16 keys need no lo part), n-tiles 0, 1 = tokens 0-7, 8-15
        float sc[2][4], sx[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[n][e] = 0.0f;
            sx[n][e] = 0.0f;
          }
        const int ltok = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row address of this lane
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int ch = 2 * kk + (lane >> 4);
          uint32_t b[4];  // (tokens 0-7 | 8-15) x (channels 16kk..+7 | +8..+15)
          ldsm_x4(b, Kr + ltok * D + ((ch ^ (ltok & 7)) * 8));
          const uint2 q2 = *reinterpret_cast<const uint2*>(qr_tab + rt_idx(0, kk, lane));
          mma_16816((kk & 1) ? sx[0] : sc[0], q2.x, 0u, q2.y, 0u, b[0], b[2]);
          mma_16816((kk & 1) ? sx[1] : sc[1], q2.x, 0u, q2.y, 0u, b[1], b[3]);
        }
        float sv[2][2];
        float tmax = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tk = 8 * n + 2 * tig + e;
            sv[n][e] = (tk < vt) ? sc[n][e] + sx[n][e] : -INFINITY;
            tmax = fmaxf(tmax, sv[n][e]);
          }
        softmax_update1(alpha * tmax);
        uint32_t ph[2], pl[2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const float pa = ex2(fmaf(sv[n][0], alpha, -m1)), pb = ex2(fmaf(sv[n][1], alpha, -m1));
          l1 += pa + pb;
          split_pair(pa, pb, ph[n], pl[n]);
        }
        // P.V: n-tile c = channels 8c..8c+7 (natural order), values by ldmatrix.trans
#pragma unroll
        for (int c = 0; c < NEV; c += 2) {
          const int ch = c + (lane >> 4);
          uint32_t b[4];  // (tokens 0-7 | 8-15) x (channel chunk c | c + 1)
          ldsm_x4_t(b, Vr + ltok * D + ((ch ^ (ltok & 7)) * 8));
          mma_16816(acc2[c], ph[0], pl[0], ph[1], pl[1], b[0], b[1]);
          mma_16816(acc2[c + 1], ph[0], pl[0], ph[1], pl[1], b[2], b[3]);
        }
      } else if (!kT && r_item) {
        // ============ residual tile: 16 FP16 tokens (chunk-swizzled rows)
        if (!in_res) {
          if (has_q) {
            // park the quantized-token part (quantized channel map) in wo
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const float vbt = reduce_over_g(vb[j]);
              vb[j] = 0.0f;
              const int h = 4 * j + tig;
              float* dd = wo + (warp * H + h) * D;
#pragma unroll
              for (int mt = 0; mt < MTV; ++mt) {
                const float fs = 16777216.0f / static_cast<float>(1 << value_pos<VB, D>(mt));
                const int c0 = vq_channel<VB, D>(g, mt, 0), c1 = vq_channel<VB, D>(g, mt, 1);
                if (c0 >= 0) dd[wo_chan<false>(h, c0)] = fmaf(acc[mt][j][0] + acc[mt][j][1], fs, vbt);
                if (c1 >= 0) dd[wo_chan<false>(h, c1)] = fmaf(acc[mt][j][2] + acc[mt][j][3], fs, vbt);
              }
#pragma unroll
              for (int mt = 0; mt < MTA; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.0f;
              if (g == 0) dm[warp * H + h] = m[j];
            }
            dumped = true;
          }
          in_res = true;
        }
        const __half* Kr = reinterpret_cast<const __half*>(stg + warp * cr);
        const __half* Vr = Kr + kResTile * D;
        const int left = r - tile * kResTile;
        const int vt = left < kResTile ? left : kResTile;

        float sc[NT][4], sx[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[j][e] = 0.0f;
            sx[j][e] = 0.0f;
          }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int ch = 2 * kk + (lane >> 4);
          uint32_t a[4];
          ldsm_x4(a, Kr + tok * D + ((ch ^ (tok & 7)) * 8));
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const uint2 bq2 = *reinterpret_cast<const uint2*>(qr_tab + rt_idx(j, kk, lane));
            mma_16816((kk & 1) ? sx[j] : sc[j], a[0], a[1], a[2], a[3], bq2.x, bq2.y);
          }
        }
        float sa[NT], sb[NT], tmax[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          sa[j] = (g < vt) ? (sc[j][0] + sx[j][0]) + (sc[j][1] + sx[j][1]) : -INFINITY;
          sb[j] = (g + 8 < vt) ? (sc[j][2] + sx[j][2]) + (sc[j][3] + sx[j][3]) : -INFINITY;
          tmax[j] = alpha * fmaxf(sa[j], sb[j]);
        }
        softmax_update(tmax);
        uint32_t b01[NT], b23[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float pa = ex2(fmaf(sa[j], alpha, -m[j])), pb = ex2(fmaf(sb[j], alpha, -m[j]));
          l[j] += pa + pb;
          uint32_t hi, lo;
          split_pair(pa, pb, hi, lo);
          pv_b(hi, lo, 8 * tig + (g >> 1), 4, b01[j], b23[j]);  // tokens (2tig, 2tig+1 | +8, +9)
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int mq = lane >> 3, rq = lane & 7;
          const int tok = rq + 8 * (mq >> 1);
          const int ch = 2 * mt + (mq & 1);
          uint32_t a[4];
          ldsm_x4_t(a, Vr + tok * D + ((ch ^ (tok & 7)) * 8));
#pragma unroll
          for (int j = 0; j < NT; ++j) mma_16816(acc[mt][j], a[0], a[1], a[2], a[3], b01[j], b23[j]);
        }
      }

      // release the consumed item's ring space (if not done yet), then refill
      if (!released) release_slot();
    }
    si = 0;

    // ---------------- warp -> shared memory
    // (a parked quantized part, already in wo, is rescaled to the final max)
    if (dumped) __syncwarp();
    if constexpr (kT) {
      float lt = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      float vbt = vb1 + __shfl_xor_sync(0xffffffffu, vb1, 1);
      vbt += __shfl_xor_sync(0xffffffffu, vbt, 2);
      if (tig == 0) {
        wm[warp * H + g] = m1;
        wl[warp * H + g] = lt;
      }
      float* oo = wo + (warp * H + g) * D;
      const float fd = dumped ? ex2(dm[warp * H + g] - m1) : 0.0f;
#pragma unroll
      for (int c = 0; c < NEV; ++c) {
        const float fs = 16777216.0f / static_cast<float>(1 << value_pos<VB, D>(c % KS));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float o = acc2[c][e] + acc2[c][e + 2];
          if (in_res) {
            const int ch = wo_chan<true>(g, 8 * c + 2 * tig + e);
            oo[ch] = dumped ? fmaf(oo[ch], fd, o) : o;
          } else {
            oo[wo_chan<true>(g, (2 * tig + e) * (D / 8) + c)] = fmaf(o, fs, vbt);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < (kT ? 0 : NT); ++j) {
      const float lt = reduce_over_g(l[j]);
      const float vbt = reduce_over_g(vb[j]);
      const int h = 4 * j + tig;
      if (g == 0) {
        wm[warp * H + h] = m[j];
        wl[warp * H + h] = lt;
      }
      float* oo = wo + (warp * H + h) * D;
      const float fd = dumped ? ex2(dm[warp * H + h] - m[j]) : 0.0f;
      if (in_res) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const float o0 = acc[mt][j][0] + acc[mt][j][1], o1 = acc[mt][j][2] + acc[mt][j][3];
          const int w0 = wo_chan<false>(h, 16 * mt + g), w1 = wo_chan<false>(h, 16 * mt + 8 + g);
          oo[w0] = dumped ? fmaf(oo[w0], fd, o0) : o0;
          oo[w1] = dumped ? fmaf(oo[w1], fd, o1) : o1;
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < MTV; ++mt) {
          const float fs = 16777216.0f / static_cast<float>(1 << value_pos<VB, D>(mt));
          const int c0 = vq_channel<VB, D>(g, mt, 0), c1 = vq_channel<VB, D>(g, mt, 1);
          if (c0 >= 0) oo[wo_chan<false>(h, c0)] = fmaf(acc[mt][j][0] + acc[mt][j][1], fs, vbt);
          if (c1 >= 0) oo[wo_chan<false>(h, c1)] = fmaf(acc[mt][j][2] + acc[mt][j][3], fs, vbt);
        }
      }
    }
    __syncthreads();

    // ---------------- CTA merge of the warps, then output or partial
    const int pf = owner_of(item_start(u, 0)), pl = owner_of(item_start(u, NI - 1));
    const int nparts = pl - pf + 1;
    const int64_t qrow = (static_cast<int64_t>(b) * p.kv_heads + kvh) * p.gqa;  // first query head row
    const int stride_slot = p.gqa * (D + 2);
    float* slot = p.partials + static_cast<int64_t>(pid + u) * stride_slot;
    // (debug builds: a partial slot outside the cache buffer is recorded and not written)
    const bool slot_ok = nparts == 1 || in_range(slot, static_cast<size_t>(stride_slot) * 4, p.partials, p.part_hi, p.err);
    for (int idx = tid; idx < p.gqa * D && slot_ok; idx += TH) {
      const int h = idx / D, c = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w * H + h]);
      float O = 0.0f, Lsum = 0.0f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float mw = wm[w * H + h];
        if (mw == -INFINITY) continue;
        const float f = ex2(mw - M);
        O += wo[(w * H + h) * D + wo_chan<kT>(h, c)] * f;
        Lsum += wl[w * H + h] * f;
      }
      if (nparts == 1) {
        p.out[(qrow + h) * D + c] = O / Lsum;
      } else {
        slot[h * D + c] = O;
        if (c == 0) {
          slot[p.gqa * D + 2 * h] = M;
          slot[p.gqa * D + 2 * h + 1] = Lsum;
        }
      }
    }
    if (nparts > 1) {
      // the last CTA of the unit to arrive merges every split's partial
      __syncthreads();
      if (tid == 0) {
        const int prev = atomic_add_acq_rel(p.counters + u, 1);
        flags[8] = (prev == nparts - 1) ? 1 : 0;
      }
      __syncthreads();
      if (flags[8]) {
        // one pass over the splits with a running (max, sum, output) per
        // element; a split's loads do not depend on the running values, so
        // the loads of several splits are in flight together
        constexpr int PER = H * D / TH;
        const int nout = p.gqa * D;
        float Mr[PER], Lr[PER], Or[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          Mr[k] = -INFINITY;
          Lr[k] = 0.0f;
          Or[k] = 0.0f;
        }
#pragma unroll 4
        for (int sidx = pf; sidx <= pl; ++sidx) {
          const float* ps = p.partials + static_cast<int64_t>(sidx + u) * stride_slot;
          if (!in_range(ps, static_cast<size_t>(stride_slot) * 4, p.partials, p.part_hi, p.err)) continue;  // debug builds
#pragma unroll
          for (int k = 0; k < PER; ++k) {
            const int idx = tid + k * TH;
            if (idx < nout) {
              const int h = idx / D;
              const float ms = __ldcg(ps + nout + 2 * h), ls = __ldcg(ps + nout + 2 * h + 1);
              const float os = __ldcg(ps + idx);
              const float mn = fmaxf(Mr[k], ms);
              const float fa = ex2(Mr[k] - mn), fb = ex2(ms - mn);
              Or[k] = fmaf(Or[k], fa, os * fb);
              Lr[k] = fmaf(Lr[k], fa, ls * fb);
              Mr[k] = mn;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          const int idx = tid + k * TH;
          if (idx < nout) p.out[qrow * D + idx] = Or[k] / Lr[k];
        }
        if (tid == 0) p.counters[u] = 0;
      }
    }
    __syncthreads();
  }
}

}  // namespace kvq
