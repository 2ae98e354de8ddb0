// Device-side building blocks shared by the append and decode kernels:
// inline-PTX wrappers (bulk TMA copies, mbarriers with bounded waits,
// warp-level tensor-core MMA, ldmatrix), the streaming-state arithmetic and
// the kernel parameter blocks.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace kvq {

// ---------------------------------------------------------------- constants

constexpr int kResTile = 16;           // residual tokens per decode work item
constexpr uint32_t kWaitLimit = 1u << 22;  // bounded mbarrier waits

// device error codes (written to the error word, never trapped)
constexpr int32_t kErrWaitTimeout = 1;
constexpr int32_t kErrBadState = 2;
constexpr int32_t kErrBadAddress = 3;  // debug builds: a computed access fell outside its buffer

// ---------------------------------------------------------------- state

// Window state of one (batch, kv head) unit of a layer: `nq` tokens held as
// quantized key groups, the rest of the appended tokens in the FP16 window,
// and the window bound (R_l at first).  After appending n tokens to T:
//   * a single-token (decode) append that brings the window to the bound on
//     a layer with an RPC ratio of rpc percent first shrinks the bound to
//     G * max(1, floor(rpc * bound / (100 G))) (KVmix, 关键设计 3:
//     num_RPC = floor(r x current_RPC), the full-precision window shrinking
//     as decoding proceeds);
//   * then the oldest G window tokens are quantized while the window holds
//     the bound or more ("LLM 量化精读笔记 · 08", section 6.2: segment, then
//     quantize).
// The bound and R_l are multiples of G, so every group starts at a multiple
// of G.  The host mirror and the single-token append kernel both step the
// state with this function.
struct WindowState {
  int64_t nq;
  int32_t bound;
};
__host__ __device__ __forceinline__ WindowState window_after_append(int64_t T, WindowState s, int n, int G,
                                                                    int rpc) {
  const int64_t r = T + n - s.nq;
  int64_t b = s.bound;
  if (n == 1 && rpc > 0 && r >= b) {
    const int64_t k = (static_cast<int64_t>(rpc) * b) / (100LL * G);
    b = static_cast<int64_t>(G) * (k > 1 ? k : 1);
  }
  WindowState o;
  o.nq = s.nq + (r >= b ? static_cast<int64_t>(G) * ((r - b) / G + 1) : 0);
  o.bound = static_cast<int32_t>(b);
  return o;
}

// ---------------------------------------------------------------- params

struct AppendParams {
  const __half* K;        // [units][n][D]
  const __half* V;
  int n;                  // tokens appended by this call
  int units;              // batch * kv heads
  int G, R;               // key group; ring slots (the window's first bound, R_l)
  int rpc;                // RPC ratio in percent (0: static window)
  // multi-token appends: the state before the call (host mirror) and the
  // quantized tokens after it; single-token appends read the state per unit
  int T0, nq0, nq1;
  int rec_bytes;
  int key_mode;           // 0: keys per channel over each group; 1: keys per token
  int64_t unit_rec_stride;   // bytes
  uint8_t* records;
  __half* res_k;          // [units][R][D] ring (chunk-swizzled)
  __half* res_v;
  int64_t res_stride;     // elements between units' rings
  int32_t* tokens;        // device state per unit: tokens appended so far,
  int32_t* nq;            //   tokens held as quantized groups,
  int32_t* bound;         //   the window bound
  int32_t* done_ctr;      // last-CTA counter of this launch
  int32_t* err;
  int mode;               // kFlush | kResidual | kUpdateState
  int ctas;               // CTAs in this launch (for the last-CTA count)
  const uint8_t* buf_lo;  // the cache buffer [buf_lo, buf_hi) (checked in debug builds)
  const uint8_t* buf_hi;
};
constexpr int kFlush = 1, kResidual = 2, kUpdateState = 4;

// Stored position of channel ch in a group record's per-channel key scale row
// and zero row (2-, 4- and 8-bit keys; 3-bit keys keep channel order).  The
// rows are kept in 8-channel chunks with chunk j of each of the four channel
// quarters side by side (position 4j + t holds chunk t*D/32 + j): decode lanes
// own one quarter each, and their four chunk loads of one instruction then
// fall in four different bank groups.  The 3-bit decode path reads single
// channels of 11-channel words, which gains nothing from the order.
__host__ __device__ constexpr int kscale_chunk_pos(int c, int D) { return (c % (D / 32)) * 4 + c / (D / 32); }
__host__ __device__ constexpr int kscale_pos(int ch, int D) { return kscale_chunk_pos(ch >> 3, D) * 8 + (ch & 7); }

// XOR applied to the word index inside token row t (within its record) of a
// record's code rows.  Rows of 128 or 64 bytes would otherwise put the rows a
// warp reads at once on the same banks: 8-bit keys at 32 words a row swap the
// 16-byte halves of each 32-byte block on odd rows; values at 16 words a row
// swap the row's 32-byte halves when t & 2; values at 32 words a row XOR the
// 32-byte block index with t & 3.  Shorter rows are stored as packed.
__host__ __device__ constexpr int code_word_xor(int words, bool key, int t) {
  return key ? (words == 32 ? (t & 1) << 2 : 0) : (words == 16 ? (t & 2) << 2 : (words == 32 ? (t & 3) << 3 : 0));
}
// one CTA per unit (a single-token append): each CTA reads and advances its
// own unit's counter, no cross-CTA handshake
constexpr int kPerUnit = 8;

struct DecodeParams {
  const __half* q;        // [B][Hq][D]
  float* out;             // [B][Hq][D]
  const uint8_t* records;
  int64_t unit_rec_stride;
  const __half* res_k;
  const __half* res_v;
  int64_t res_stride;     // elements
  const int32_t* tokens;  // device state: unit 0's appended-token counter (all units agree)
  const int32_t* nq;      //   and its quantized-token counter
  float* partials;        // [slots][gqa][D + 2]
  int32_t* counters;      // [units]
  int32_t* err;
  int units;
  int kv_heads;
  int gqa;                // query heads per kv head
  int G, R;               // key group; ring slots
  int rec_bytes;
  int grid;               // CTAs launched
  float alpha;            // log2(e) / sqrt(D)
  const uint8_t* buf_lo;  // the cache buffer [buf_lo, buf_hi) (checked in debug builds)
  const uint8_t* buf_hi;
  const uint8_t* part_hi; // end of the partials buffer (checked in debug builds)
  // launch mode: 0 ordinary; 1 programmatic dependent that waits for the
  // previous kernel of the stream before its first read; 2 programmatic
  // dependent that stages its first cache items before that wait (only where
  // the previous kernel writes neither this layer's cache nor its counters)
  int pdl;
};

struct ChunkParams {
  const __half* q;        // [B][Hq][n][D]: queries of the n newest tokens
  float* out;             // [B][Hq][n][D]
  const uint8_t* records;
  int64_t unit_rec_stride;
  const __half* res_k;
  const __half* res_v;
  int64_t res_stride;     // elements
  int32_t* err;
  int n;                  // queries per (batch, head)
  int T;                  // tokens appended so far
  int n_q;                // tokens held as quantized groups
  int Hq, kv_heads, gqa;
  int qpb;                // queries per CTA: 128 / gqa
  int G, R;
  int gshift;             // log2(G)
  int kb, vb, km;
  int wk, wv;             // u32 words per key / value code row
  int rec_bytes;
  int off_kscale;         // record offset of the key (scale, zero) part
  int off_vsz;            // record offset of the value (scale, zero) pairs
  float alpha;            // log2(e) / sqrt(D)
  uint8_t* ws;            // workspace: dequantized tiles, ws_tiles per unit
  int ws_tiles;
  const uint8_t* ws_hi;   // end of the workspace (checked in debug builds)
  const uint8_t* buf_lo;  // the cache buffer [buf_lo, buf_hi) (checked in debug builds)
  const uint8_t* buf_hi;
};

// ---------------------------------------------------------------- debug checks

// Debug builds (compiled with KVQ_DEBUG) check that [p, p + bytes) lies in
// [lo, hi) before a computed access; a failed check records kErrBadAddress
// in the error word and the caller skips the access.  Release builds
// compile the check to `true`.
__device__ __forceinline__ bool in_range(const void* p, size_t bytes, const void* lo, const void* hi, int32_t* err) {
#ifdef KVQ_DEBUG
  const uint8_t* a = static_cast<const uint8_t*>(p);
  if (a >= static_cast<const uint8_t*>(lo) && a + bytes <= static_cast<const uint8_t*>(hi)) return true;
  atomicExch(err, kErrBadAddress);
  return false;
#else
  (void)p; (void)bytes; (void)lo; (void)hi; (void)err;
  return true;
#endif
}

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Atomic add with acquire-release semantics at gpu scope: the release makes
// the CTA's earlier writes (ordered before it by a CTA barrier) visible to
// whoever acquires the counter later; the acquire does the converse.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch.  grid_dep_launch lets the next kernel of the
// stream (if launched as a programmatic dependent) start its CTAs while this
// grid still runs; grid_dep_wait returns once the previous kernel of the
// stream has completed and its memory writes are visible.  Both are no-ops
// for an ordinary launch.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// make generic-proxy shared-memory writes visible to the async (TMA) proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// one arrival on an mbarrier (release: earlier writes are visible to its waiters)
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completion signalled on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy shared -> global (bulk-group completion).
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// the shared-memory sources of all committed bulk stores have been read
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Bounded wait on an mbarrier phase.  Returns false (and records the error)
// if the phase did not complete within `limit` tries.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase, int32_t* err, uint32_t limit = kWaitLimit) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(phase)
        : "memory");
    if (done) return true;
  }
  atomicExch(err, kErrWaitTimeout);
  return false;
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (x & mask) | magic in one LOP3
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(magic));
  return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// e holds two fp16 values 1024 + 2^k * code (exact); returns the codes, exact:
// e * 2^-k - 1024 * 2^-k with one fma.  The constants are built from their
// fp16 bit patterns so they fold at compile time.
__device__ __forceinline__ uint32_t magic_fix(uint32_t e, int k) {
  const uint32_t sc = static_cast<uint32_t>(15 - k) << 10;                // 2^-k
  const uint32_t of = 0x8000u | (static_cast<uint32_t>(25 - k) << 10);   // -1024 * 2^-k
  return h2_as_u32(__hfma2(u32_as_h2(e), u32_as_h2(sc | (sc << 16)), u32_as_h2(of | (of << 16))));
}

// 2^x for x <= 0 (probabilities and rescale factors), one MUFU op
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr uint32_t kMagic = 0x64006400u;  // fp16 1024.0 in both halves

}  // namespace kvq
