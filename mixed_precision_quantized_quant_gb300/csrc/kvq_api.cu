// Host side of the C ABI declared in include/kvq.h: configuration checks,
// cache layout inside the caller's buffer, the per-layer dispatch table, the
// host mirror of the streaming state, launches and the graph-replayed decode
// step.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/kvq.h"
#include "kvq_kernels.h"

namespace {

// NVTX range around a C-ABI call (a no-op unless a profiler is attached)
struct Trace {
  explicit Trace(const char* name) { nvtxRangePushA(name); }
  ~Trace() { nvtxRangePop(); }
};

using kvq::AppendParams;
using kvq::DecodeParams;

constexpr int kMaxGrid = 1024;       // decode CTAs per launch (bounds the partial buffer)
constexpr int64_t kAlign = 256;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int words_per_row(int d, int b) { return b == 3 ? (d + 10) / 11 : d * b / 32; }
bool bits_ok(int b) { return b == 2 || b == 3 || b == 4 || b == 8; }

struct LayerPlan {
  int kb, vb, R;  // R: ring slots, the window's first bound
  int rpc;        // RPC ratio in percent (0: static window)
  int km;  // key mode: 0 per channel over key groups, 1 per token
  int wk, wv;
  int64_t rec_bytes;
  int64_t max_groups;
  int64_t unit_rec_stride;
  int64_t off_records, off_res_k, off_res_v;
  int64_t res_stride_elems;
};

struct Plan {
  int L, B, Hq, Hkv, D, G, max_tokens, gqa, units;
  std::vector<LayerPlan> layers;
  int64_t off_ctrl, ctrl_stride, off_err, off_counters, off_partials, partial_floats;
  int64_t total;
};

kvq_status make_plan(const kvq_config* cfg, Plan* P) {
  if (!cfg || !cfg->layers) return KVQ_ERR_ARG;
  if (cfg->num_layers < 1 || cfg->batch < 1 || cfg->num_q_heads < 1 || cfg->num_kv_heads < 1 ||
      cfg->max_tokens < 1)
    return KVQ_ERR_ARG;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return KVQ_ERR_ARG;
  if (cfg->group_size != 32 && cfg->group_size != 64 && cfg->group_size != 128) return KVQ_ERR_ARG;
  if (cfg->num_q_heads % cfg->num_kv_heads != 0) return KVQ_ERR_ARG;
  const int gqa = cfg->num_q_heads / cfg->num_kv_heads;
  if (gqa > 8) return KVQ_ERR_UNSUPPORTED;
  P->L = cfg->num_layers;
  P->B = cfg->batch;
  P->Hq = cfg->num_q_heads;
  P->Hkv = cfg->num_kv_heads;
  P->D = cfg->head_dim;
  P->G = cfg->group_size;
  P->max_tokens = cfg->max_tokens;
  P->gqa = gqa;
  P->units = cfg->batch * cfg->num_kv_heads;
  int64_t off = 0;
  // per layer: {append done-counter, padding to 64 B, then per unit: appended
  // tokens, quantized tokens, window bound}
  P->ctrl_stride = align_up(64 + 3 * static_cast<int64_t>(P->units) * 4, kAlign);
  P->off_ctrl = off;
  off += P->ctrl_stride * P->L;
  P->off_err = off;
  off += kAlign;
  P->off_counters = off;
  off += align_up(static_cast<int64_t>(P->units) * 4, kAlign);
  P->partial_floats = static_cast<int64_t>(kMaxGrid + P->units) * gqa * (P->D + 2);
  P->off_partials = off;
  off += align_up(P->partial_floats * 4, kAlign);
  P->layers.clear();
  for (int l = 0; l < P->L; ++l) {
    const kvq_layer_cfg& lc = cfg->layers[l];
    if (lc.rpc_percent > 100) return KVQ_ERR_ARG;
    if (!bits_ok(lc.k_bits) || !bits_ok(lc.v_bits)) return KVQ_ERR_BITS;
    if (lc.key_mode != KVQ_KEY_PER_CHANNEL && lc.key_mode != KVQ_KEY_PER_TOKEN) return KVQ_ERR_ARG;
    if (lc.key_mode == KVQ_KEY_PER_TOKEN && lc.k_bits == 3) return KVQ_ERR_UNSUPPORTED;
    if (lc.residual < P->G || lc.residual % P->G != 0) return KVQ_ERR_ARG;
    LayerPlan lp;
    lp.kb = lc.k_bits;
    lp.vb = lc.v_bits;
    lp.R = lc.residual;
    lp.rpc = lc.rpc_percent;
    lp.wk = words_per_row(P->D, lp.kb);
    lp.wv = words_per_row(P->D, lp.vb);
    lp.km = lc.key_mode;
    // key scale/zero: d pairs of rows per group (per channel) or one pair per token
    lp.rec_bytes = 4LL * P->G * (lp.wk + lp.wv) + (lp.km ? 4LL * P->G : 4LL * P->D) + 4LL * P->G;
    lp.max_groups = P->max_tokens / P->G;
    {
      // the decode kernel splits a layer's work in 32-bit byte-cost units
      const int64_t slice = 4LL * 32 * (lp.wk + lp.wv) + (lp.km ? 128LL : 4LL * P->D) + 128;
      const int64_t tile = 16LL * 4 * P->D;
      const int64_t setup = 16 * (slice > 2048 ? slice : 2048);  // 2 x up to 8 warps per CTA
      // (stages round up to whole records and tiles: one stage of each more)
      const int64_t per_unit = setup + lp.max_groups * (P->G / 32) * slice + ((lp.R + 15) / 16) * tile +
                               8 * slice + 8 * tile;
      if (per_unit * P->units >= (1LL << 32)) return KVQ_ERR_UNSUPPORTED;
    }
    lp.unit_rec_stride = align_up(lp.max_groups * lp.rec_bytes, kAlign);
    lp.off_records = off;
    off += lp.unit_rec_stride * P->units;
    lp.res_stride_elems = static_cast<int64_t>(lp.R) * P->D;
    lp.off_res_k = off;
    off += align_up(lp.res_stride_elems * 2 * P->units, kAlign);
    lp.off_res_v = off;
    off += align_up(lp.res_stride_elems * 2 * P->units, kAlign);
    P->layers.push_back(lp);
  }
  P->total = off;
  return KVQ_OK;
}

struct StepGraph {
  std::vector<const void*> key;
  cudaGraphExec_t exec = nullptr;
  // capture helpers: the appends run on a forked stream, each decode waits
  // for its own layer's append only
  cudaStream_t aux = nullptr;
  std::vector<cudaEvent_t> ev;  // [0]: fork, [1 + l]: append of layer l done
};

}  // namespace

struct kvq_handle {
  Plan plan;
  int device = 0;  // the device current at kvq_create (the buffer's device)
  uint8_t* base = nullptr;
  // host mirror of each layer's window state (every unit of a layer agrees)
  std::vector<int64_t> tokens;  // appended tokens
  std::vector<int64_t> nq;      // tokens held as quantized groups
  std::vector<int32_t> bound;   // window bound
  std::vector<kvq::DecodeKernel> dec;
  std::vector<int> grid;
  std::vector<int> app_grid;  // persistent CTAs of a prefill flush launch
  StepGraph graph;
};

namespace {

int32_t* ctrl(kvq_handle* h, int layer) {
  return reinterpret_cast<int32_t*>(h->base + h->plan.off_ctrl + static_cast<int64_t>(layer) * h->plan.ctrl_stride);
}
// per-unit counters of a layer: appended tokens (16 ints past its
// done-counter), then quantized tokens, then the window bound
int32_t* unit_tokens(kvq_handle* h, int layer) { return ctrl(h, layer) + 16; }
int32_t* unit_nq(kvq_handle* h, int layer) { return unit_tokens(h, layer) + h->plan.units; }
int32_t* unit_bound(kvq_handle* h, int layer) { return unit_nq(h, layer) + h->plan.units; }

// The layer's window state after appending n tokens (host mirror).
kvq::WindowState mirror_after(const kvq_handle* h, int layer, int n) {
  kvq::WindowState w;
  w.nq = h->nq[layer];
  w.bound = h->bound[layer];
  return kvq::window_after_append(h->tokens[layer], w, n, h->plan.G, h->plan.layers[layer].rpc);
}
void mirror_advance(kvq_handle* h, int layer, int n) {
  const kvq::WindowState w = mirror_after(h, layer, n);
  h->tokens[layer] += n;
  h->nq[layer] = w.nq;
  h->bound[layer] = w.bound;
}
int32_t* errw(kvq_handle* h) { return reinterpret_cast<int32_t*>(h->base + h->plan.off_err); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq_status launch_append(kvq_handle* h, int layer, const void* K, const void* V, int n, cudaStream_t s) {
  const Plan& P = h->plan;
  const LayerPlan& lp = P.layers[layer];
  const int64_t T = h->tokens[layer];
  const int64_t nq0 = h->nq[layer];
  const int64_t nq1 = mirror_after(h, layer, n).nq;
  const int64_t nflush = (nq1 - nq0) / P.G;
  const int64_t first_res = T > nq1 ? T : nq1;
  const int64_t nres = T + n - first_res;

  AppendParams ap;
  ap.K = static_cast<const __half*>(K);
  ap.V = static_cast<const __half*>(V);
  ap.n = n;
  ap.units = P.units;
  ap.G = P.G;
  ap.R = lp.R;
  ap.rpc = lp.rpc;
  ap.T0 = static_cast<int>(T);
  ap.nq0 = static_cast<int>(nq0);
  ap.nq1 = static_cast<int>(nq1);
  ap.rec_bytes = static_cast<int>(lp.rec_bytes);
  ap.key_mode = lp.km;
  ap.unit_rec_stride = lp.unit_rec_stride;
  ap.records = h->base + lp.off_records;
  ap.res_k = reinterpret_cast<__half*>(h->base + lp.off_res_k);
  ap.res_v = reinterpret_cast<__half*>(h->base + lp.off_res_v);
  ap.res_stride = lp.res_stride_elems;
  ap.tokens = unit_tokens(h, layer);
  ap.nq = unit_nq(h, layer);
  ap.bound = unit_bound(h, layer);
  ap.done_ctr = ctrl(h, layer);
  ap.err = errw(h);
  ap.buf_lo = h->base;
  ap.buf_hi = h->base + P.total;
  const size_t smem = kvq::append_smem_bytes(lp.kb, lp.vb, P.D, P.G, static_cast<int>(lp.rec_bytes));
  cudaError_t e = cudaSuccess;
  if (n == 1) {
    // one CTA per unit: its flush jobs (if the window reaches its bound) and its new token
    ap.mode = kvq::kFlush | kvq::kResidual | kvq::kUpdateState | kvq::kPerUnit;
    ap.ctas = P.units;
    e = kvq::append_dispatch(lp.kb, lp.vb, P.D, ap, dim3(P.units, 1), kvq::append_block_threads(lp.kb, lp.vb, P.G), smem, s);
  } else {
    if (nflush > 0) {
      const int64_t jobs = nflush * P.units;
      const int ctas = static_cast<int>(jobs < h->app_grid[layer] ? jobs : h->app_grid[layer]);
      ap.mode = kvq::kFlush | (nres == 0 ? kvq::kUpdateState : 0);
      ap.ctas = ctas;
      e = kvq::append_dispatch(lp.kb, lp.vb, P.D, ap, dim3(static_cast<unsigned>(ctas), 1),
                               kvq::append_block_threads(lp.kb, lp.vb, P.G), smem, s);
    }
    if (e == cudaSuccess && nres > 0) {
      const int64_t chunks = (nres + 15) / 16;
      ap.mode = kvq::kResidual | kvq::kUpdateState;
      ap.ctas = static_cast<int>(chunks * P.units);
      e = kvq::append_dispatch(lp.kb, lp.vb, P.D, ap, dim3(static_cast<unsigned>(chunks), P.units), 128, 0, s);
    }
  }
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  mirror_advance(h, layer, n);
  return KVQ_OK;
}

// Launches the layer's decode kernel.  pdl (see DecodeParams::pdl): 0 an
// ordinary launch, 1 or 2 a programmatic dependent of the previous kernel of
// the stream, so that its CTAs launch while that kernel drains.
kvq_status launch_decode(kvq_handle* h, int layer, const void* q, float* out, cudaStream_t s, int pdl) {
  const Plan& P = h->plan;
  const LayerPlan& lp = P.layers[layer];
  DecodeParams dp;
  dp.q = static_cast<const __half*>(q);
  dp.out = out;
  dp.records = h->base + lp.off_records;
  dp.unit_rec_stride = lp.unit_rec_stride;
  dp.res_k = reinterpret_cast<const __half*>(h->base + lp.off_res_k);
  dp.res_v = reinterpret_cast<const __half*>(h->base + lp.off_res_v);
  dp.res_stride = lp.res_stride_elems;
  dp.tokens = unit_tokens(h, layer);
  dp.nq = unit_nq(h, layer);
  dp.partials = reinterpret_cast<float*>(h->base + P.off_partials);
  dp.counters = reinterpret_cast<int32_t*>(h->base + P.off_counters);
  dp.err = errw(h);
  dp.units = P.units;
  dp.kv_heads = P.Hkv;
  dp.gqa = P.gqa;
  dp.G = P.G;
  dp.R = lp.R;
  dp.rec_bytes = static_cast<int>(lp.rec_bytes);
  dp.grid = h->grid[layer];
  dp.alpha = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(P.D)));
  dp.buf_lo = h->base;
  dp.buf_hi = h->base + P.total;
  dp.part_hi = reinterpret_cast<const uint8_t*>(dp.partials) + P.partial_floats * 4;
  dp.pdl = pdl;
  const kvq::DecodeKernel& k = h->dec[layer];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(h->grid[layer]));
  cfg.blockDim = dim3(static_cast<unsigned>(k.threads));
  cfg.dynamicSmemBytes = k.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, k.fn, dp) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

// Tiles of one unit in the chunk workspace: the quantized part and the
// window part each start a new 64-token tile.
int64_t chunk_ws_tiles(const Plan& P) { return (P.max_tokens + 63) / 64 + 1; }

kvq_status launch_chunk(kvq_handle* h, int layer, const void* q, int n, float* out, void* ws, cudaStream_t s) {
  const Plan& P = h->plan;
  const LayerPlan& lp = P.layers[layer];
  kvq::ChunkParams cp;
  cp.q = static_cast<const __half*>(q);
  cp.out = out;
  cp.records = h->base + lp.off_records;
  cp.unit_rec_stride = lp.unit_rec_stride;
  cp.res_k = reinterpret_cast<const __half*>(h->base + lp.off_res_k);
  cp.res_v = reinterpret_cast<const __half*>(h->base + lp.off_res_v);
  cp.res_stride = lp.res_stride_elems;
  cp.err = errw(h);
  cp.n = n;
  cp.T = static_cast<int>(h->tokens[layer]);
  cp.n_q = static_cast<int>(h->nq[layer]);
  cp.Hq = P.Hq;
  cp.kv_heads = P.Hkv;
  cp.gqa = P.gqa;
  cp.qpb = kvq::chunk_queries_per_cta(P.gqa);
  cp.G = P.G;
  cp.R = lp.R;
  cp.gshift = P.G == 32 ? 5 : P.G == 64 ? 6 : 7;
  cp.kb = lp.kb;
  cp.vb = lp.vb;
  cp.km = lp.km;
  cp.wk = lp.wk;
  cp.wv = lp.wv;
  cp.rec_bytes = static_cast<int>(lp.rec_bytes);
  cp.off_kscale = static_cast<int>(4LL * P.G * (lp.wk + lp.wv));
  cp.off_vsz = cp.off_kscale + static_cast<int>(lp.km ? 4LL * P.G : 4LL * P.D);
  cp.alpha = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(P.D)));
  cp.ws = static_cast<uint8_t*>(ws);
  cp.ws_tiles = static_cast<int>(chunk_ws_tiles(P));
  cp.ws_hi = cp.ws + static_cast<int64_t>(P.units) * cp.ws_tiles * static_cast<int64_t>(kvq::chunk_tile_bytes(P.D));
  cp.buf_lo = h->base;
  cp.buf_hi = h->base + P.total;
  const int tiles = (cp.n_q + 63) / 64 + (cp.T - cp.n_q + 63) / 64;
  if (kvq::chunk_attn_launch(lp.kb, lp.vb, P.D, cp, P.units, tiles, s) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

// A wait that nothing completes: the bounded wait of every kernel must give
// up, record kErrWaitTimeout in the error word and return (no trap, no hang).
__global__ void bounded_wait_selftest_kernel(int32_t* err, uint32_t limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    kvq::mbar_init(&bar, 1);
    kvq::fence_mbar_init();
  }
  __syncthreads();
  kvq::mbar_wait(&bar, 0, err, limit);  // no arrival ever comes
}

}  // namespace

extern "C" {

size_t kvq_cache_bytes(const kvq_config* cfg) {
  Plan P;
  if (make_plan(cfg, &P) != KVQ_OK) return 0;
  return static_cast<size_t>(P.total);
}

kvq_status kvq_create(const kvq_config* cfg, void* dev_buf, size_t bytes, kvq_handle** out) {
  Trace trace("kvq_create");
  if (!out) return KVQ_ERR_ARG;
  *out = nullptr;
  Plan P;
  kvq_status st = make_plan(cfg, &P);
  if (st != KVQ_OK) return st;
  if (!dev_buf) return KVQ_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_buf) & (kAlign - 1)) != 0) return KVQ_ERR_ALIGN;
  if (bytes < static_cast<size_t>(P.total)) return KVQ_ERR_CAPACITY;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVQ_ERR_CUDA;
  kvq_handle* h = new (std::nothrow) kvq_handle;
  if (!h) return KVQ_ERR_ARG;
  h->plan = P;
  h->device = dev;
  h->base = static_cast<uint8_t*>(dev_buf);
  h->tokens.assign(P.L, 0);
  h->nq.assign(P.L, 0);
  h->bound.assign(P.L, 0);
  for (int l = 0; l < P.L; ++l) h->bound[l] = P.layers[l].R;
  for (int l = 0; l < P.L; ++l) {
    const LayerPlan& lp = P.layers[l];
    kvq::DecodeKernel k = kvq::decode_select(lp.kb, lp.vb, P.D, P.gqa, lp.km);
    if (!k.fn) {
      delete h;
      return KVQ_ERR_UNSUPPORTED;
    }
    h->dec.push_back(k);
    int gsz = sms * k.ctas_per_sm;
    if (gsz > kMaxGrid) gsz = kMaxGrid;
    h->grid.push_back(gsz);
    const size_t asmem = kvq::append_smem_bytes(lp.kb, lp.vb, P.D, P.G, static_cast<int>(lp.rec_bytes));
    const int aocc = kvq::append_ctas_per_sm(lp.kb, lp.vb, P.D, P.G, kvq::append_block_threads(lp.kb, lp.vb, P.G), asmem);
    if (aocc < 1) {
      delete h;
      return KVQ_ERR_UNSUPPORTED;
    }
    h->app_grid.push_back(sms * aocc);
  }
  // zero everything, then set every unit's window bound to its layer's R_l
  std::vector<int32_t> ctrl_init(static_cast<size_t>(P.ctrl_stride * P.L / 4), 0);
  for (int l = 0; l < P.L; ++l)
    for (int u = 0; u < P.units; ++u)
      ctrl_init[static_cast<size_t>(l * P.ctrl_stride / 4 + 16 + 2 * P.units + u)] = P.layers[l].R;
  if (cudaMemset(dev_buf, 0, static_cast<size_t>(P.total)) != cudaSuccess ||
      cudaMemcpy(h->base + P.off_ctrl, ctrl_init.data(), ctrl_init.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    delete h;
    return KVQ_ERR_CUDA;
  }
  *out = h;
  return KVQ_OK;
}

kvq_status kvq_append(kvq_handle* h, int layer, const void* K, const void* V, int n_tokens, void* stream) {
  Trace trace("kvq_append");
  if (!h || layer < 0 || layer >= h->plan.L || n_tokens < 0) return KVQ_ERR_ARG;
  if (n_tokens == 0) return KVQ_OK;
  if (!K || !V) return KVQ_ERR_ARG;
  if (!aligned16(K) || !aligned16(V)) return KVQ_ERR_ALIGN;
  if (h->tokens[layer] + n_tokens > h->plan.max_tokens) return KVQ_ERR_CAPACITY;
  return launch_append(h, layer, K, V, n_tokens, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_decode_attn(kvq_handle* h, int layer, const void* q, float* out, void* stream) {
  Trace trace("kvq_decode_attn");
  if (!h || layer < 0 || layer >= h->plan.L) return KVQ_ERR_ARG;
  if (!q || !out) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_ALIGN;
  if (h->tokens[layer] <= 0) return KVQ_ERR_STATE;
  return launch_decode(h, layer, q, out, static_cast<cudaStream_t>(stream), 1);
}

size_t kvq_chunk_workspace_bytes(const kvq_handle* h) {
  if (!h) return 0;
  return static_cast<size_t>(h->plan.units) * static_cast<size_t>(chunk_ws_tiles(h->plan)) *
         kvq::chunk_tile_bytes(h->plan.D);
}

kvq_status kvq_chunk_attn(kvq_handle* h, int layer, const void* q, int n_queries, float* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  Trace trace("kvq_chunk_attn");
  if (!h || layer < 0 || layer >= h->plan.L) return KVQ_ERR_ARG;
  if (!q || !out || !workspace) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return KVQ_ERR_ALIGN;
  if (workspace_bytes < kvq_chunk_workspace_bytes(h)) return KVQ_ERR_CAPACITY;
  if (h->tokens[layer] <= 0) return KVQ_ERR_STATE;
  if (n_queries < 1 || n_queries > h->tokens[layer]) return KVQ_ERR_ARG;
  if (kvq::chunk_queries_per_cta(h->plan.gqa) < 1 || h->plan.units > 65535) return KVQ_ERR_UNSUPPORTED;
  return launch_chunk(h, layer, q, n_queries, out, workspace, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_decode_step(kvq_handle* h, const void* const* K, const void* const* V, const void* const* q,
                           float* const* out, void* stream) {
  Trace trace("kvq_decode_step");
  if (!h || !K || !V || !q || !out) return KVQ_ERR_ARG;
  const int L = h->plan.L;
  for (int l = 0; l < L; ++l) {
    if (!K[l] || !V[l] || !q[l] || !out[l]) return KVQ_ERR_ARG;
    if (!aligned16(K[l]) || !aligned16(V[l]) || !aligned16(q[l]) || !aligned16(out[l])) return KVQ_ERR_ALIGN;
    if (h->tokens[l] + 1 > h->plan.max_tokens) return KVQ_ERR_CAPACITY;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<const void*> key;
  key.reserve(4 * L);
  for (int l = 0; l < L; ++l) {
    key.push_back(K[l]);
    key.push_back(V[l]);
    key.push_back(q[l]);
    key.push_back(out[l]);
  }
  if (s == nullptr) {  // the legacy stream cannot be captured: launch directly
    for (int l = 0; l < L; ++l) {
      kvq_status st = launch_append(h, l, K[l], V[l], 1, s);
      if (st != KVQ_OK) return st;
      st = launch_decode(h, l, q[l], out[l], s, 1);
      if (st != KVQ_OK) return st;
    }
    return KVQ_OK;
  }
  if (!h->graph.exec || h->graph.key != key) {
    if (h->graph.exec) {
      cudaGraphExecDestroy(h->graph.exec);
      h->graph.exec = nullptr;
    }
    const std::vector<int64_t> saved_t = h->tokens, saved_q = h->nq;
    const std::vector<int32_t> saved_b = h->bound;
    if (!h->graph.aux) {
      if (cudaStreamCreateWithFlags(&h->graph.aux, cudaStreamNonBlocking) != cudaSuccess) return KVQ_ERR_CUDA;
      h->graph.ev.assign(L + 1, nullptr);
      for (auto& e : h->graph.ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return KVQ_ERR_CUDA;
    }
    cudaStream_t a = h->graph.aux;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return KVQ_ERR_CUDA;
    kvq_status st = KVQ_OK;
    // appends of all layers on the forked stream (they touch only their own
    // layer's records, ring and counters); decode l waits for append l and
    // runs after decode l-1 (they share the split workspace).  Decode l is a
    // programmatic dependent of decode l-1, which writes nothing of layer l's
    // cache: it stages its first cache items while decode l-1 drains, and
    // reads the query and touches the workspace only after decode l-1 is done.
    if (cudaEventRecord(h->graph.ev[0], s) != cudaSuccess || cudaStreamWaitEvent(a, h->graph.ev[0], 0) != cudaSuccess)
      st = KVQ_ERR_CUDA;
    for (int l = 0; l < L && st == KVQ_OK; ++l) {
      st = launch_append(h, l, K[l], V[l], 1, a);
      if (st == KVQ_OK && cudaEventRecord(h->graph.ev[1 + l], a) != cudaSuccess) st = KVQ_ERR_CUDA;
    }
    for (int l = 0; l < L && st == KVQ_OK; ++l) {
      if (cudaStreamWaitEvent(s, h->graph.ev[1 + l], 0) != cudaSuccess) st = KVQ_ERR_CUDA;
      if (st == KVQ_OK) st = launch_decode(h, l, q[l], out[l], s, 2);
    }
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(s, &graph);
    h->tokens = saved_t;
    h->nq = saved_q;
    h->bound = saved_b;
    if (st != KVQ_OK || ec != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return st != KVQ_OK ? st : KVQ_ERR_CUDA;
    }
    const cudaError_t ei = cudaGraphInstantiate(&h->graph.exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) {
      h->graph.exec = nullptr;
      return KVQ_ERR_CUDA;
    }
    h->graph.key = key;
  }
  if (cudaGraphLaunch(h->graph.exec, s) != cudaSuccess) return KVQ_ERR_CUDA;
  for (int l = 0; l < L; ++l) mirror_advance(h, l, 1);
  return KVQ_OK;
}

kvq_status kvq_layer_view_get(const kvq_handle* h, int layer, kvq_layer_view* v) {
  if (!h || !v || layer < 0 || layer >= h->plan.L) return KVQ_ERR_ARG;
  const Plan& P = h->plan;
  const LayerPlan& lp = P.layers[layer];
  std::memset(v, 0, sizeof(*v));
  v->k_bits = lp.kb;
  v->v_bits = lp.vb;
  v->residual = lp.R;
  v->group_size = P.G;
  v->head_dim = P.D;
  v->k_words = lp.wk;
  v->v_words = lp.wv;
  v->key_mode = lp.km;
  v->record_bytes = lp.rec_bytes;
  v->unit_record_stride = lp.unit_rec_stride;
  v->residual_stride = lp.res_stride_elems * 2;
  v->tokens = h->tokens[layer];
  v->quantized_tokens = h->nq[layer];
  v->residual_tokens = v->tokens - v->quantized_tokens;
  v->window_bound = h->bound[layer];
  v->rpc_percent = lp.rpc;
  v->records = h->base + lp.off_records;
  v->residual_k = h->base + lp.off_res_k;
  v->residual_v = h->base + lp.off_res_v;
  return KVQ_OK;
}

double kvq_equivalent_bits(const kvq_handle* h) {
  if (!h) return 0.0;
  double s = 0.0;
  for (const LayerPlan& lp : h->plan.layers) s += 0.5 * (lp.kb + lp.vb);
  return s / h->plan.L;
}

int64_t kvq_decode_bytes(const kvq_handle* h, int layer) {
  if (!h || layer < 0 || layer >= h->plan.L) return -1;
  const Plan& P = h->plan;
  const LayerPlan& lp = P.layers[layer];
  const int64_t T = h->tokens[layer];
  const int64_t nq = h->nq[layer];
  const int64_t r = T - nq;
  const int64_t per_unit = (nq / P.G) * lp.rec_bytes + r * 4LL * P.D;
  return P.units * per_unit + static_cast<int64_t>(P.B) * P.Hq * P.D * (2 + 4);
}

kvq_status kvq_device_error(kvq_handle* h, int32_t* code, void* stream) {
  Trace trace("kvq_device_error");
  if (!h || !code) return KVQ_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, errw(h), 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
  *code = v;
  if (v != 0 && cudaMemset(errw(h), 0, 4) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_selftest_bounded_wait(kvq_handle* h, void* stream) {
  Trace trace("kvq_selftest_bounded_wait");
  if (!h) return KVQ_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t before = 0;
  kvq_status st = kvq_device_error(h, &before, stream);  // start from a clear error word
  if (st != KVQ_OK) return st;
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(errw(h), 4096u);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  int32_t code = 0;
  st = kvq_device_error(h, &code, stream);  // synchronizes, reads and clears
  if (st != KVQ_OK) return st;
  return code == kvq::kErrWaitTimeout ? KVQ_OK : KVQ_ERR_STATE;
}

namespace {

// Bytes of the counters region and of one layer's window ring (keys then
// values, adjacent in the buffer) in a snapshot.
int64_t ctrl_bytes(const Plan& P) { return P.ctrl_stride * P.L; }
int64_t ring_bytes(const Plan& P, const LayerPlan& lp) {
  return lp.off_res_v - lp.off_res_k + align_up(lp.res_stride_elems * 2 * P.units, kAlign);
}

}  // namespace

size_t kvq_state_bytes(const kvq_handle* h) {
  if (!h) return 0;
  int64_t n = ctrl_bytes(h->plan);
  for (const LayerPlan& lp : h->plan.layers) n += ring_bytes(h->plan, lp);
  return static_cast<size_t>(n);
}

kvq_status kvq_state_save(kvq_handle* h, void* dst, void* stream) {
  Trace trace("kvq_state_save");
  if (!h || !dst) return KVQ_ERR_ARG;
  if (!aligned16(dst)) return KVQ_ERR_ALIGN;
  const Plan& P = h->plan;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* d = static_cast<uint8_t*>(dst);
  if (cudaMemcpyAsync(d, h->base + P.off_ctrl, ctrl_bytes(P), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  d += ctrl_bytes(P);
  for (const LayerPlan& lp : P.layers) {
    if (cudaMemcpyAsync(d, h->base + lp.off_res_k, ring_bytes(P, lp), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return KVQ_ERR_CUDA;
    d += ring_bytes(P, lp);
  }
  return KVQ_OK;
}

kvq_status kvq_state_restore(kvq_handle* h, const void* src, void* stream) {
  Trace trace("kvq_state_restore");
  if (!h || !src) return KVQ_ERR_ARG;
  if (!aligned16(src)) return KVQ_ERR_ALIGN;
  const Plan& P = h->plan;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<int32_t> c(static_cast<size_t>(ctrl_bytes(P) / 4));
  if (cudaMemcpyAsync(c.data(), src, ctrl_bytes(P), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  std::vector<int64_t> tokens(P.L), nq(P.L);
  std::vector<int32_t> bound(P.L);
  for (int l = 0; l < P.L; ++l) {
    const LayerPlan& lp = P.layers[l];
    const int32_t* cl = c.data() + l * P.ctrl_stride / 4;
    if (cl[0] != 0) return KVQ_ERR_STATE;  // an append's last-CTA counter mid-launch
    const int32_t t = cl[16], q = cl[16 + P.units], b = cl[16 + 2 * P.units];
    for (int u = 1; u < P.units; ++u)
      if (cl[16 + u] != t || cl[16 + P.units + u] != q || cl[16 + 2 * P.units + u] != b) return KVQ_ERR_STATE;
    if (q < 0 || q % P.G != 0 || q > t || t > P.max_tokens) return KVQ_ERR_STATE;
    if (b < P.G || b > lp.R || b % P.G != 0 || (lp.rpc == 0 && b != lp.R)) return KVQ_ERR_STATE;
    if (t - q >= b) return KVQ_ERR_STATE;
    tokens[l] = t;
    nq[l] = q;
    bound[l] = b;
  }
  const uint8_t* d = static_cast<const uint8_t*>(src);
  if (cudaMemcpyAsync(h->base + P.off_ctrl, d, ctrl_bytes(P), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  d += ctrl_bytes(P);
  for (const LayerPlan& lp : P.layers) {
    if (cudaMemcpyAsync(h->base + lp.off_res_k, d, ring_bytes(P, lp), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return KVQ_ERR_CUDA;
    d += ring_bytes(P, lp);
  }
  h->tokens = tokens;
  h->nq = nq;
  h->bound = bound;
  return KVQ_OK;
}

kvq_status kvq_destroy(kvq_handle* h) {
  Trace trace("kvq_destroy");
  if (!h) return KVQ_ERR_ARG;
  for (cudaEvent_t e : h->graph.ev)
    if (e) cudaEventDestroy(e);
  if (h->graph.aux) cudaStreamDestroy(h->graph.aux);
  if (h->graph.exec) cudaGraphExecDestroy(h->graph.exec);
  delete h;
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_ARG: return "invalid argument";
    case KVQ_ERR_BITS: return "bit width outside {2,3,4,8}";
    case KVQ_ERR_ALIGN: return "pointer not aligned";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_STATE: return "invalid state";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

}  // extern "C"

// ------------------------------------------------------- allocation-free decode
//
// kvq_decode_attn_noalloc(): the decode kernel with its split-merge workspace
// in a static device array instead of the caller's cache buffer.  Host code
// only sees a stand-in symbol for the array, so each device's real address is
// looked up once with cudaGetSymbolAddress and kept.

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
uint8_t* g_noalloc_ptr[kMaxDevices] = {};

// The array's address on `dev`, which must be the current device (host code
// sees the array only through a stand-in symbol; the runtime resolves it for
// the current device).
kvq_status noalloc_scratch(int dev, uint8_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_noalloc(kvq_handle* h, int layer, const void* q, float* out,
                                              void* stream) {
  Trace trace("kvq_decode_attn_noalloc");
  if (!h || layer < 0 || layer >= h->plan.L) return KVQ_ERR_ARG;
  if (!q || !out) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_ALIGN;
  if (h->tokens[layer] <= 0) return KVQ_ERR_STATE;
  const Plan& P = h->plan;
  const LayerPlan& lp = P.layers[layer];
  const int grid = h->grid[layer];
  const int64_t counter_bytes = align_up(static_cast<int64_t>(P.units) * 4, 256);
  const int64_t partial_bytes = static_cast<int64_t>(grid + P.units) * P.gqa * (P.D + 2) * 4;
  if (counter_bytes + partial_bytes > static_cast<int64_t>(KVQ_NOALLOC_SCRATCH_BYTES)) return KVQ_ERR_CAPACITY;
  // the array is looked up (and the kernel launched) on the device that holds
  // the handle's buffer: a different current device is refused
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cur != h->device) return KVQ_ERR_ARG;
  uint8_t* scratch = nullptr;
  const kvq_status st = noalloc_scratch(cur, &scratch);
  if (st != KVQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* counters = reinterpret_cast<int32_t*>(scratch);
  if (cudaMemsetAsync(counters, 0, static_cast<size_t>(P.units) * 4, s) != cudaSuccess) return KVQ_ERR_CUDA;
  DecodeParams dp;
  dp.q = static_cast<const __half*>(q);
  dp.out = out;
  dp.records = h->base + lp.off_records;
  dp.unit_rec_stride = lp.unit_rec_stride;
  dp.res_k = reinterpret_cast<const __half*>(h->base + lp.off_res_k);
  dp.res_v = reinterpret_cast<const __half*>(h->base + lp.off_res_v);
  dp.res_stride = lp.res_stride_elems;
  dp.tokens = unit_tokens(h, layer);
  dp.nq = unit_nq(h, layer);
  dp.partials = reinterpret_cast<float*>(scratch + counter_bytes);
  dp.counters = counters;
  dp.err = errw(h);
  dp.units = P.units;
  dp.kv_heads = P.Hkv;
  dp.gqa = P.gqa;
  dp.G = P.G;
  dp.R = lp.R;
  dp.rec_bytes = static_cast<int>(lp.rec_bytes);
  dp.grid = grid;
  dp.alpha = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(P.D)));
  dp.buf_lo = h->base;
  dp.buf_hi = h->base + P.total;
  dp.part_hi = reinterpret_cast<const uint8_t*>(dp.partials) + partial_bytes;
  dp.pdl = 0;
  const kvq::DecodeKernel& k = h->dec[layer];
  k.fn<<<grid, k.threads, k.smem, s>>>(dp);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}
