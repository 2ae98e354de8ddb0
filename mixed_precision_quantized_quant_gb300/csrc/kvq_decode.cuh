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

constexpr int kStages = 2;

__host__ __device__ constexpr int dec_stage_bytes(int D, int rec_bytes) {
  return (((rec_bytes > kResTile * 4 * D) ? rec_bytes : kResTile * 4 * D) + 127) / 128 * 128;
}

struct DecodeSmem {
  int stage_bytes;
  int off_bars, off_qs, off_qp, off_qr, off_wm, off_wl, off_dm, off_flags, off_wo, off_dump, total;
};

__host__ __device__ inline DecodeSmem decode_smem_layout(int D, int NT, int rec_bytes) {
  DecodeSmem s;
  const int H = 4 * NT;
  s.stage_bytes = dec_stage_bytes(D, rec_bytes);
  int off = kWarps * kStages * s.stage_bytes;
  s.off_bars = off;
  off += kWarps * kStages * 8;
  s.off_qs = off;
  off += H * D * 2;
  s.off_qp = off;
  off += 32 * (NT * D / 8 + 4) * 4;
  s.off_qr = off;
  off += 32 * (NT * D / 16 * 2 + 4) * 4;
  s.off_wm = off;
  off += kWarps * H * 4;
  s.off_wl = off;
  off += kWarps * H * 4;
  s.off_dm = off;
  off += kWarps * H * 4;
  s.off_flags = off;
  off += 64;
  off = (off + 15) / 16 * 16;
  s.off_wo = off;
  off += kWarps * H * D * 4;
  s.off_dump = off;
  off += kWarps * H * D * 4;
  s.total = off;
  return s;
}

// ------------------------------------------------------------------ unpacking

// Code pairs of one key word, in the order the query pairs are built:
//  4-bit: (c0,c4) (c1,c5) (c2,c6) (c3,c7); 2-bit: (c_i, c_{8+i}), i = 0..7;
//  8-bit: (c0,c2) (c1,c3).  Each pair is a half2 of exact integer codes.
template <int KB>
__device__ __forceinline__ void k_word_pairs(uint32_t w, uint32_t* e) {
  if constexpr (KB == 4) {
    const uint32_t t = w >> 8;
    e[0] = magic_fix(and_or(w, 0x000F000Fu, kMagic), 1.0f);
    e[1] = magic_fix(and_or(w, 0x00F000F0u, kMagic), 1.0f / 16.0f);
    e[2] = magic_fix(and_or(t, 0x000F000Fu, kMagic), 1.0f);
    e[3] = magic_fix(and_or(t, 0x00F000F0u, kMagic), 1.0f / 16.0f);
  } else if constexpr (KB == 2) {
    const uint32_t t = w >> 10;
#pragma unroll
    for (int i = 0; i < 5; ++i)
      e[i] = magic_fix(and_or(w, 0x00030003u << (2 * i), kMagic), 1.0f / static_cast<float>(1 << (2 * i)));
#pragma unroll
    for (int i = 0; i < 3; ++i)
      e[5 + i] = magic_fix(and_or(t, 0x00030003u << (2 * i), kMagic), 1.0f / static_cast<float>(1 << (2 * i)));
  } else {  // 8-bit
    e[0] = magic_fix(prmt(w, 0x64646464u, 0x4240u), 1.0f);
    e[1] = magic_fix(prmt(w, 0x64646464u, 0x4341u), 1.0f);
  }
}

// Channel pair (ca, cb) of pair e of a key word starting at channel cbase.
template <int KB>
__device__ __forceinline__ void k_pair_channels(int cbase, int e, int& ca, int& cb) {
  ca = cbase + e;
  cb = cbase + e + (KB == 4 ? 4 : (KB == 2 ? 8 : 2));
}

// 2-bit field i (0..7) of both halves of x -> half2 of exact codes
__device__ __forceinline__ uint32_t f2(uint32_t x, int i) {
  if (i < 5) return magic_fix(and_or(x, 0x00030003u << (2 * i), kMagic), 1.0f / static_cast<float>(1 << (2 * i)));
  return magic_fix(and_or(x >> 10, 0x00030003u << (2 * (i - 5)), kMagic),
                   1.0f / static_cast<float>(1 << (2 * (i - 5))));
}
__device__ __forceinline__ uint32_t f4(uint32_t x, int f) {
  const uint32_t y = (f >= 2) ? (x >> 8) : x;
  return (f & 1) ? magic_fix(and_or(y, 0x00F000F0u, kMagic), 1.0f / 16.0f)
                 : magic_fix(and_or(y, 0x000F000Fu, kMagic), 1.0f);
}
__device__ __forceinline__ uint32_t f8(uint32_t z, int i) {
  return magic_fix(and_or(i ? (z >> 8) : z, 0x00FF00FFu, kMagic), 1.0f);
}

// Value code pairs for two tokens (a, b): H[c] = (code_a[c], code_b[c]) for the
// D/8 channels this thread owns.  wa/wb hold the thread's slice of each row.
template <int VB, int D>
__device__ __forceinline__ void v_pairs(const uint32_t* wa, const uint32_t* wb, uint32_t half_sel,
                                        uint32_t (&H)[D / 8]) {
  if constexpr (VB == 2) {
    if constexpr (D == 128) {
      const uint32_t x = prmt(wa[0], wb[0], 0x5410u), y = prmt(wa[0], wb[0], 0x7632u);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        H[i] = f2(x, i);
        H[8 + i] = f2(y, i);
      }
    } else {
      const uint32_t x = prmt(wa[0], wb[0], half_sel);
#pragma unroll
      for (int i = 0; i < 8; ++i) H[i] = f2(x, i);
    }
  } else if constexpr (VB == 4) {
#pragma unroll
    for (int k = 0; k < D / 64; ++k) {
      const uint32_t x = prmt(wa[k], wb[k], 0x5410u), y = prmt(wa[k], wb[k], 0x7632u);
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        H[8 * k + f] = f4(x, f);
        H[8 * k + 4 + f] = f4(y, f);
      }
    }
  } else {  // 8-bit
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      const uint32_t z = prmt(wa[k], wb[k], 0x5410u), y = prmt(wa[k], wb[k], 0x7632u);
      H[4 * k] = f8(z, 0);
      H[4 * k + 1] = f8(z, 1);
      H[4 * k + 2] = f8(y, 0);
      H[4 * k + 3] = f8(y, 1);
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

__device__ __forceinline__ float reduce_over_g(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// ------------------------------------------------------------------ kernel

template <int KB, int VB, int D, int NT>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeParams p) {
  constexpr int NP = D / 8;      // key pairs per token row per thread = value channels per thread
  constexpr int KS = D / 16;     // k-steps of q.K^T = channel m-tiles of p.V
  constexpr int WK = D * KB / 32;
  constexpr int WT = WK / 4;     // key words per thread per row
  constexpr int PW = 16 / KB;    // pairs per key word
  constexpr int WV = D * VB / 32;
  constexpr int VW = (D * VB / 256) > 0 ? (D * VB / 256) : 1;  // value words per thread per row
  constexpr int H = 4 * NT;      // padded query heads
  constexpr int QPS = NT * NP + 4;
  constexpr int QRS = NT * KS * 2 + 4;

  extern __shared__ __align__(128) uint8_t smem[];
  const DecodeSmem L = decode_smem_layout(D, NT, p.rec_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bars);
  __half* qs = reinterpret_cast<__half*>(smem + L.off_qs);
  uint32_t* qp_tab = reinterpret_cast<uint32_t*>(smem + L.off_qp);
  uint32_t* qr_tab = reinterpret_cast<uint32_t*>(smem + L.off_qr);
  float* wm = reinterpret_cast<float*>(smem + L.off_wm);
  float* wl = reinterpret_cast<float*>(smem + L.off_wl);
  float* dm = reinterpret_cast<float*>(smem + L.off_dm);
  int* flags = reinterpret_cast<int*>(smem + L.off_flags);
  float* wo = reinterpret_cast<float*>(smem + L.off_wo);
  float* dump = reinterpret_cast<float*>(smem + L.off_dump);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tig = lane & 3, part = g & 1;

  // ---------------- state and this CTA's share of the work
  const int64_t T = __ldcg(p.tokens);
  if (T <= 0) return;
  const int64_t nq = quantized_after(T, p.R, p.G);
  const int64_t r = T - nq;
  const int64_t NG = nq / p.G;
  const int64_t NRT = (r + kResTile - 1) / kResTile;
  const int64_t NI = NG + NRT;
  const int64_t cq = p.rec_bytes, cr = static_cast<int64_t>(kResTile) * 4 * D;
  const int64_t Cu = NG * cq + NRT * cr;
  const int64_t C = static_cast<int64_t>(p.units) * Cu;
  const int64_t maxc = (NRT > 0 && cr > cq) || NG == 0 ? cr : cq;
  int64_t peff = C / maxc;
  if (peff < 1) peff = 1;
  if (peff > p.grid) peff = p.grid;
  const int64_t pid = blockIdx.x;
  if (pid >= peff) return;

  auto item_start = [&](int64_t f) -> int64_t {
    const int64_t u = f / NI, i = f % NI;
    return u * Cu + (i < NG ? i * cq : NG * cq + (i - NG) * cr);
  };
  auto first_item_at = [&](int64_t x) -> int64_t {  // first flat item starting at or after x
    const int64_t u = x / Cu, o = x - u * Cu;
    int64_t i;
    if (o == 0) {
      i = 0;
    } else if (NG > 0 && o <= (NG - 1) * cq) {
      i = (o + cq - 1) / cq;
    } else if (o <= NG * cq) {
      i = NG;
    } else {
      i = NG + (o - NG * cq + cr - 1) / cr;
    }
    return u * NI + i;
  };
  auto owner = [&](int64_t f) -> int64_t { return (item_start(f) * peff) / C; };
  const int64_t f0 = first_item_at((pid * C + peff - 1) / peff);
  const int64_t f1 = first_item_at(((pid + 1) * C + peff - 1) / peff);

  // ---------------- pipeline setup (warp-private stages)
  uint8_t* stage_base = smem + warp * kStages * L.stage_bytes;
  uint64_t* wbar = bars + warp * kStages;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&wbar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int64_t f, int st) {
    const int64_t u = f / NI, i = f % NI;
    uint8_t* dst = stage_base + st * L.stage_bytes;
    fence_proxy_async_smem();
    if (i < NG) {
      mbar_arrive_expect_tx(&wbar[st], static_cast<uint32_t>(p.rec_bytes));
      bulk_g2s(dst, p.records + u * p.unit_rec_stride + i * p.rec_bytes, static_cast<uint32_t>(p.rec_bytes),
               &wbar[st]);
    } else {
      const int64_t k = i - NG;
      const int64_t slot0 = (nq + k * kResTile) % p.R;
      const uint32_t bytes = kResTile * D * 2;
      mbar_arrive_expect_tx(&wbar[st], 2 * bytes);
      bulk_g2s(dst, p.res_k + u * p.res_stride + slot0 * D, bytes, &wbar[st]);
      bulk_g2s(dst + bytes, p.res_v + u * p.res_stride + slot0 * D, bytes, &wbar[st]);
    }
  };

  int64_t k_item = 0;  // this warp's item counter
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) {
      const int64_t f = f0 + warp + 4 * s;
      if (f < f1) issue(f, s);
    }
  }

  const __half2 negmask = part ? __float2half2_rn(-1.0f) : __float2half2_rn(0.0f);
  const float alpha = p.alpha;
  const uint32_t vhalf_sel = (g & 1) ? 0x7632u : 0x5410u;  // 2-bit values, D = 64
  const int64_t u_first = f0 / NI, u_last = (f1 - 1) / NI;

  for (int64_t u = u_first; u <= u_last; ++u) {
    const int64_t seg_hi = ((u + 1) * NI < f1) ? (u + 1) * NI : f1;
    const int b = static_cast<int>(u / p.kv_heads), kvh = static_cast<int>(u % p.kv_heads);

    // ---------------- per-unit query tables
    for (int idx = tid; idx < H * D / 2; idx += kThreads) {
      const int h = idx / (D / 2), c2 = idx % (D / 2);
      __half2 v = __float2half2_rn(0.0f);
      if (h < p.gqa)
        v = reinterpret_cast<const __half2*>(p.q + (static_cast<int64_t>(b) * p.kv_heads * p.gqa +
                                                    static_cast<int64_t>(kvh) * p.gqa + h) * D)[c2];
      reinterpret_cast<__half2*>(qs)[idx] = v;
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t* qp = qp_tab + lane * QPS;
      uint32_t* qr = qr_tab + lane * QRS;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int h = 4 * j + (g >> 1);
        const bool live = h < p.gqa;
        for (int pi = 0; pi < NP; ++pi) {
          const int wi = pi / PW, e = pi % PW;
          int ca, cb;
          k_pair_channels<KB>(tig * (D / 4) + wi * (32 / KB), e, ca, cb);
          qp[j * NP + pi] = live ? h2_as_u32(__halves2half2(qs[h * D + ca], qs[h * D + cb])) : 0u;
        }
        for (int kk = 0; kk < KS; ++kk) {
          for (int rr = 0; rr < 2; ++rr) {
            const int c = 16 * kk + 8 * rr + 2 * tig;
            qr[(j * KS + kk) * 2 + rr] =
                (live && !part) ? h2_as_u32(__halves2half2(qs[h * D + c], qs[h * D + c + 1])) : 0u;
          }
        }
      }
    }
    __syncthreads();

    // ---------------- warp state for this unit
    float m[NT], l[NT], vb[NT];
    float acc[KS][NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.0f;
      vb[j] = 0.0f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.0f;
    }
    bool has_q = false, in_res = false, dumped = false;

    // online-softmax update for one tile of 16 tokens (scores already scaled)
    auto softmax_tile = [&](float (&sa)[NT], float (&sb)[NT]) {
      float tmax[NT];
      bool need = false;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float t = fmaxf(sa[j], sb[j]);
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 4));
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 8));
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 16));
        tmax[j] = t;
        need |= t > m[j] + 8.0f;
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float mn = fmaxf(m[j], tmax[j]);
          const float f = (mn == -INFINITY) ? 1.0f : exp2f(m[j] - mn);
          m[j] = mn;
          l[j] *= f;
          vb[j] *= f;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][j][e] *= f;
        }
      }
    };

    while (true) {
      const int64_t f = f0 + warp + 4 * k_item;
      if (f >= seg_hi) break;
      const int st = static_cast<int>(k_item % kStages);
      const uint32_t ph = static_cast<uint32_t>((k_item / kStages) & 1);
      if (!mbar_wait(&wbar[st], ph, p.err)) return;
      const uint8_t* stg = stage_base + st * L.stage_bytes;
      const int64_t i = f % NI;

      if (i < NG) {
        // ============ quantized group
        has_q = true;
        const uint32_t* Kc = reinterpret_cast<const uint32_t*>(stg);
        const uint32_t* Vc = Kc + p.G * WK;
        const __half* Ks = reinterpret_cast<const __half*>(Vc + p.G * WV);
        const __half* Kz = Ks + D;
        const __half2* Vsz = reinterpret_cast<const __half2*>(Kz + D);

        uint32_t qp[NT][NP];
        {
          const uint32_t* src = qp_tab + lane * QPS;
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int pi = 0; pi < NP; pi += 4) {
              const uint4 v = *reinterpret_cast<const uint4*>(src + j * NP + pi);
              qp[j][pi] = v.x;
              qp[j][pi + 1] = v.y;
              qp[j][pi + 2] = v.z;
              qp[j][pi + 3] = v.w;
            }
        }
        // zero pairs -> bias = sum_c q_c z_c, one MMA per k-step (zeros broadcast over rows)
        float bias[NT];
        {
          uint32_t zn[NP];
          const uint32_t* zsrc = reinterpret_cast<const uint32_t*>(Kz + tig * (D / 4));
#pragma unroll
          for (int pi = 0; pi < NP; pi += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(zsrc + pi);
            zn[pi] = v.x;
            zn[pi + 1] = v.y;
            zn[pi + 2] = v.z;
            zn[pi + 3] = v.w;
          }
          uint32_t zp[NP];
#pragma unroll
          for (int wi = 0; wi < WT; ++wi) {
            const uint32_t* nn = zn + wi * PW;  // natural pairs of this word's channels
            uint32_t* oo = zp + wi * PW;
            if constexpr (KB == 4) {
              oo[0] = prmt(nn[0], nn[2], 0x5410u);
              oo[1] = prmt(nn[0], nn[2], 0x7632u);
              oo[2] = prmt(nn[1], nn[3], 0x5410u);
              oo[3] = prmt(nn[1], nn[3], 0x7632u);
            } else if constexpr (KB == 2) {
#pragma unroll
              for (int kq = 0; kq < 4; ++kq) {
                oo[2 * kq] = prmt(nn[kq], nn[kq + 4], 0x5410u);
                oo[2 * kq + 1] = prmt(nn[kq], nn[kq + 4], 0x7632u);
              }
            } else {
              oo[0] = prmt(nn[0], nn[1], 0x5410u);
              oo[1] = prmt(nn[0], nn[1], 0x7632u);
            }
          }
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              mma_16816(c, zp[2 * kk], zp[2 * kk], zp[2 * kk + 1], zp[2 * kk + 1], qp[j][2 * kk], qp[j][2 * kk + 1]);
            bias[j] = c[0];
          }
        }
        // folded query q~ = q * s, hi part in even columns, lo part in odd ones
        uint32_t bq[NT][NP];
        {
          uint32_t sn[NP];
          const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(Ks + tig * (D / 4));
#pragma unroll
          for (int pi = 0; pi < NP; pi += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(ssrc + pi);
            sn[pi] = v.x;
            sn[pi + 1] = v.y;
            sn[pi + 2] = v.z;
            sn[pi + 3] = v.w;
          }
#pragma unroll
          for (int wi = 0; wi < WT; ++wi) {
            const uint32_t* nn = sn + wi * PW;
            uint32_t sp[PW];
            if constexpr (KB == 4) {
              sp[0] = prmt(nn[0], nn[2], 0x5410u);
              sp[1] = prmt(nn[0], nn[2], 0x7632u);
              sp[2] = prmt(nn[1], nn[3], 0x5410u);
              sp[3] = prmt(nn[1], nn[3], 0x7632u);
            } else if constexpr (KB == 2) {
#pragma unroll
              for (int kq = 0; kq < 4; ++kq) {
                sp[2 * kq] = prmt(nn[kq], nn[kq + 4], 0x5410u);
                sp[2 * kq + 1] = prmt(nn[kq], nn[kq + 4], 0x7632u);
              }
            } else {
              sp[0] = prmt(nn[0], nn[1], 0x5410u);
              sp[1] = prmt(nn[0], nn[1], 0x7632u);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int e = 0; e < PW; ++e) {
                const __half2 qq = u32_as_h2(qp[j][wi * PW + e]);
                const __half2 ss = u32_as_h2(sp[e]);
                const __half2 hi = __hmul2(qq, ss);
                bq[j][wi * PW + e] = h2_as_u32(__hfma2(qq, ss, __hmul2(hi, negmask)));
              }
          }
        }

        for (int t0 = 0; t0 < p.G; t0 += 16) {
          // ---- scores for tokens t0+g (row g) and t0+g+8 (row g+8)
          float sc[NT][4];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            sc[j][0] = bias[j];
            sc[j][1] = 0.0f;
            sc[j][2] = bias[j];
            sc[j][3] = 0.0f;
          }
          {
            uint32_t k0[WT], k1[WT];
            lds_words<WT>(k0, Kc + (t0 + g) * WK + tig * WT);
            lds_words<WT>(k1, Kc + (t0 + g + 8) * WK + tig * WT);
#pragma unroll
            for (int wi = 0; wi < WT; ++wi) {
              uint32_t e0[PW], e1[PW];
              k_word_pairs<KB>(k0[wi], e0);
              k_word_pairs<KB>(k1[wi], e1);
#pragma unroll
              for (int e = 0; e < PW; e += 2)
#pragma unroll
                for (int j = 0; j < NT; ++j)
                  mma_16816(sc[j], e0[e], e1[e], e0[e + 1], e1[e + 1], bq[j][wi * PW + e], bq[j][wi * PW + e + 1]);
            }
          }
          float sa[NT], sb[NT];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            sa[j] = (sc[j][0] + sc[j][1]) * alpha;
            sb[j] = (sc[j][2] + sc[j][3]) * alpha;
          }
          softmax_tile(sa, sb);
          const float2 sza = __half22float2(Vsz[t0 + g]);
          const float2 szb = __half22float2(Vsz[t0 + g + 8]);
          uint32_t b01[NT], b23[NT];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const float pa = exp2f(sa[j] - m[j]), pb = exp2f(sb[j] - m[j]);
            l[j] += pa + pb;
            vb[j] = fmaf(pa, sza.y, fmaf(pb, szb.y, vb[j]));
            const float ta = pa * sza.x, tb = pb * szb.x;
            const __half2 hi = __floats2half2_rn(ta, tb);
            const __half2 lo = __floats2half2_rn(ta - __low2float(hi), tb - __high2float(hi));
            const int srcA = 4 * tig + (g >> 1), srcB = srcA + 16;
            const uint32_t xh = __shfl_sync(0xffffffffu, h2_as_u32(hi), srcA);
            const uint32_t yh = __shfl_sync(0xffffffffu, h2_as_u32(hi), srcB);
            const uint32_t xl = __shfl_sync(0xffffffffu, h2_as_u32(lo), srcA);
            const uint32_t yl = __shfl_sync(0xffffffffu, h2_as_u32(lo), srcB);
            const uint32_t x = part ? xl : xh, y = part ? yl : yh;
            b01[j] = prmt(x, y, 0x5410u);  // tokens tig, tig+4
            b23[j] = prmt(x, y, 0x7632u);  // tokens tig+8, tig+12
          }
          // ---- p~.V over tokens (tig, tig+4 | tig+8, tig+12), rows = channels
          {
            const int voff = (VB == 2 && D == 64) ? (g >> 1) : g * VW;
            uint32_t w0[VW], w1[VW], w2[VW], w3[VW];
            lds_words<VW>(w0, Vc + (t0 + tig) * WV + voff);
            lds_words<VW>(w1, Vc + (t0 + tig + 4) * WV + voff);
            lds_words<VW>(w2, Vc + (t0 + tig + 8) * WV + voff);
            lds_words<VW>(w3, Vc + (t0 + tig + 12) * WV + voff);
            uint32_t h01[NP], h23[NP];
            v_pairs<VB, D>(w0, w1, vhalf_sel, h01);
            v_pairs<VB, D>(w2, w3, vhalf_sel, h23);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
              for (int j = 0; j < NT; ++j)
                mma_16816(acc[mt][j], h01[mt], h01[KS + mt], h23[mt], h23[KS + mt], b01[j], b23[j]);
          }
        }
      } else {
        // ============ residual tile: 16 FP16 tokens (chunk-swizzled rows)
        if (!in_res) {
          if (has_q) {
            // park the quantized-token part (channel map of the quantized path)
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const float vbt = reduce_over_g(vb[j]);
              vb[j] = 0.0f;
              const int h = 4 * j + tig;
              float* dd = dump + (warp * H + h) * D;
#pragma unroll
              for (int mt = 0; mt < KS; ++mt) {
                dd[g * NP + mt] = acc[mt][j][0] + acc[mt][j][1] + vbt;
                dd[g * NP + KS + mt] = acc[mt][j][2] + acc[mt][j][3] + vbt;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.0f;
              }
              if (g == 0) dm[warp * H + h] = m[j];
            }
            dumped = true;
          }
          in_res = true;
        }
        const __half* Kr = reinterpret_cast<const __half*>(stg);
        const __half* Vr = Kr + kResTile * D;
        const int64_t kt = i - NG;
        const int64_t left = r - kt * kResTile;
        const int vt = left < kResTile ? static_cast<int>(left) : kResTile;

        float sc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[j][e] = 0.0f;
        const uint32_t* qrs = qr_tab + lane * QRS;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int ch = 2 * kk + (lane >> 4);
          uint32_t a[4];
          ldsm_x4(a, Kr + tok * D + ((ch ^ (tok & 7)) * 8));
#pragma unroll
          for (int j = 0; j < NT; ++j)
            mma_16816(sc[j], a[0], a[1], a[2], a[3], qrs[(j * KS + kk) * 2], qrs[(j * KS + kk) * 2 + 1]);
        }
        float sa[NT], sb[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          sa[j] = (g < vt) ? (sc[j][0] + sc[j][1]) * alpha : -INFINITY;
          sb[j] = (g + 8 < vt) ? (sc[j][2] + sc[j][3]) * alpha : -INFINITY;
        }
        softmax_tile(sa, sb);
        uint32_t b01[NT], b23[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float pa = exp2f(sa[j] - m[j]), pb = exp2f(sb[j] - m[j]);
          l[j] += pa + pb;
          const __half2 hi = __floats2half2_rn(pa, pb);
          const __half2 lo = __floats2half2_rn(pa - __low2float(hi), pb - __high2float(hi));
          const int srcA = 8 * tig + (g >> 1), srcB = srcA + 4;
          const uint32_t xh = __shfl_sync(0xffffffffu, h2_as_u32(hi), srcA);
          const uint32_t yh = __shfl_sync(0xffffffffu, h2_as_u32(hi), srcB);
          const uint32_t xl = __shfl_sync(0xffffffffu, h2_as_u32(lo), srcA);
          const uint32_t yl = __shfl_sync(0xffffffffu, h2_as_u32(lo), srcB);
          const uint32_t x = part ? xl : xh, y = part ? yl : yh;
          b01[j] = prmt(x, y, 0x5410u);  // tokens 2tig, 2tig+1
          b23[j] = prmt(x, y, 0x7632u);  // tokens 2tig+8, 2tig+9
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

      __syncwarp();
      if (lane == 0) {
        const int64_t fn = f + 4 * kStages;
        if (fn < f1) issue(fn, st);
      }
      ++k_item;
    }

    // ---------------- warp -> shared memory
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float lt = reduce_over_g(l[j]);
      const float vbt = reduce_over_g(vb[j]);
      const int h = 4 * j + tig;
      if (g == 0) {
        wm[warp * H + h] = m[j];
        wl[warp * H + h] = lt;
      }
      float* oo = wo + (warp * H + h) * D;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        if (in_res) {
          oo[16 * mt + g] = acc[mt][j][0] + acc[mt][j][1];
          oo[16 * mt + 8 + g] = acc[mt][j][2] + acc[mt][j][3];
        } else {
          oo[g * NP + mt] = acc[mt][j][0] + acc[mt][j][1] + vbt;
          oo[g * NP + KS + mt] = acc[mt][j][2] + acc[mt][j][3] + vbt;
        }
      }
    }
    if (lane == 0) flags[warp] = dumped ? 1 : 0;
    __syncthreads();

    // ---------------- CTA merge of the warps, then output or partial
    const int64_t pf = owner(u * NI), pl = owner(u * NI + NI - 1);
    const int nparts = static_cast<int>(pl - pf + 1);
    const int64_t qrow = (static_cast<int64_t>(b) * p.kv_heads + kvh) * p.gqa;  // first query head row
    const int stride_slot = p.gqa * (D + 2);
    float* slot = p.partials + (pid + u) * stride_slot;
    for (int idx = tid; idx < p.gqa * D; idx += kThreads) {
      const int h = idx / D, c = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * H + h]);
      float O = 0.0f, Lsum = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = wm[w * H + h];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - M);
        float o = wo[(w * H + h) * D + c];
        if (flags[w]) o += dump[(w * H + h) * D + c] * exp2f(dm[w * H + h] - mw);
        O += o * f;
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
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int prev = atomicAdd(p.counters + u, 1);
        flags[8] = (prev == nparts - 1) ? 1 : 0;
      }
      __syncthreads();
      if (flags[8]) {
        __threadfence();
        for (int idx = tid; idx < p.gqa * D; idx += kThreads) {
          const int h = idx / D, c = idx % D;
          float M = -INFINITY;
          for (int64_t s = pf; s <= pl; ++s) M = fmaxf(M, __ldcg(p.partials + (s + u) * stride_slot + p.gqa * D + 2 * h));
          float O = 0.0f, Lsum = 0.0f;
          for (int64_t s = pf; s <= pl; ++s) {
            const float* ps = p.partials + (s + u) * stride_slot;
            const float f = exp2f(__ldcg(ps + p.gqa * D + 2 * h) - M);
            O += __ldcg(ps + h * D + c) * f;
            Lsum += __ldcg(ps + p.gqa * D + 2 * h + 1) * f;
          }
          p.out[(qrow + h) * D + c] = O / Lsum;
        }
        if (tid == 0) p.counters[u] = 0;
      }
    }
    __syncthreads();
  }
}

}  // namespace kvq
