/*
 * kvq.h -- layer-wise mixed-precision KV-cache quantization and decode
 * attention over the quantized cache, for NVIDIA GB300 (sm_103a).
 *
 * The method (sources are web pages, cited by title and section):
 *   - every layer stores its cache at a static precision pair KxVy,
 *     x, y in {2, 3, 4, 8}, chosen offline and loaded with no online cost
 *     ("KVTuner: Sensitivity-Aware Layer-Wise Mixed-Precision KV Cache
 *     Quantization ...", sections A1 and A2; "KVmix: Gradient-Based Layer
 *     Importance-Aware Mixed-Precision Quantization for KV Cache", 关键设计 2 and 4);
 *   - keys are quantized asymmetrically per channel over groups of G tokens
 *     (or, per layer, per token), values per token, with scale = (max - min)/(2^b - 1), zero = min and
 *     code = clamp(rint((x - min)/scale), 0, 2^b - 1); codes are packed into
 *     32-bit words, 3-bit words holding ten 3-bit fields and one 2-bit field
 *     (KVTuner section A3 "KV缓存量化基础"; KVmix 关键设计 2; "LLM 量化精读笔记 · 08
 *     KV Cache 量化：KIVI 与误差累积", sections 6.1 and 6.2);
 *   - the most recent tokens stay in an FP16 residual window of R_l tokens;
 *     when the window holds R_l or more tokens the oldest G are quantized as one
 *     key group (KIVI notes section 6.2; KVmix 关键设计 3); with an RPC ratio
 *     (KVmix 关键设计 3, num_RPC = floor(r x current_RPC)) the window bound
 *     shrinks as decoding proceeds (see kvq_layer_cfg.rpc_percent);
 *   - decode attention a = softmax(q K^T / sqrt(d)), o = a V runs over the
 *     quantized tokens (dequantized on the fly) and the FP16 window, after the
 *     new token has been appended (KVTuner section A3 equation).
 *
 * Conventions shared by all entry points:
 *   - The library allocates no device memory.  The caller allocates one device
 *     buffer of kvq_cache_bytes() bytes and hands it to kvq_create(); the
 *     library carves the per-layer caches, their state and its workspace out
 *     of it.  The caller frees it after kvq_destroy().
 *   - Device pointers passed to kvq_append() and kvq_decode_attn() must be
 *     16-byte aligned and stay valid until the work queued on `stream` is done.
 *   - Arguments are checked on the host before anything is launched; a failed
 *     check returns a status and changes nothing.  KVQ_ERR_CUDA reports a
 *     failed launch; the handle's host-side state is then undefined.
 *   - Work is queued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and runs asynchronously.  One handle is driven by
 *     one host thread at a time; calls on a handle are ordered by the caller.
 *   - All sequences of a batch share one length.
 *   - No kernel spins without bound and none traps: a device-side wait that
 *     gives up sets an error word that kvq_device_error() reports.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_ARG = 1,      /* null pointer, bad dimension, layer out of range   */
  KVQ_ERR_BITS = 2,     /* a bit width outside {2, 3, 4, 8}                  */
  KVQ_ERR_ALIGN = 3,    /* a pointer that is not 16-byte aligned             */
  KVQ_ERR_CAPACITY = 4, /* appending past max_tokens, or buffer too small    */
  KVQ_ERR_CUDA = 5,     /* a CUDA runtime call failed                        */
  KVQ_ERR_STATE = 6,    /* call not valid now (e.g. attention on empty layer)*/
  KVQ_ERR_UNSUPPORTED = 7 /* a shape the library has no kernel for        */
} kvq_status;

/* Key quantization mode of a layer (KVTuner sections A3-A4 evaluate both):
 *   KVQ_KEY_PER_CHANNEL: keys per channel over each group of G tokens (KIVI);
 *   KVQ_KEY_PER_TOKEN:   keys per token over their head_dim channels, like
 *                        values ("per-token-asym"); k_bits in {2, 4, 8}. */
#define KVQ_KEY_PER_CHANNEL 0
#define KVQ_KEY_PER_TOKEN 1

/* One layer's static precision pair, key mode and FP16 residual window (tokens).
 * k_bits, v_bits in {2, 3, 4, 8}; residual >= group_size and a multiple of it.
 * key_mode KVQ_KEY_PER_TOKEN with k_bits = 3 is KVQ_ERR_UNSUPPORTED.
 *
 * rpc_percent (0..100; KVQ_ERR_ARG above 100) is KVmix's RPC ratio (关键设计 3:
 * num_RPC = floor(r x current_RPC), 20% on its high-precision layers, 10% on
 * the others, the full-precision count shrinking as decoding proceeds).  0
 * keeps a static window of `residual` tokens.  Otherwise the layer keeps a
 * window bound C, first `residual` (the prompt's share): any append quantizes
 * the oldest group_size window tokens while the window holds C or more, and a
 * single-token append that brings the window to C first sets
 * C = group_size * max(1, floor(rpc_percent * C / (100 * group_size))).
 * Multi-token appends keep C.  The ring keeps `residual` slots. */
typedef struct {
  uint8_t k_bits;
  uint8_t v_bits;
  uint8_t key_mode;     /* KVQ_KEY_PER_CHANNEL or KVQ_KEY_PER_TOKEN */
  uint8_t rpc_percent;  /* 0: static window; else the RPC ratio in percent */
  int32_t residual;
} kvq_layer_cfg;

/* Shape of the cache.
 *   num_q_heads % num_kv_heads == 0 and num_q_heads / num_kv_heads <= 8
 *   head_dim in {64, 128}; group_size in {32, 64, 128}
 *   max_tokens: capacity per sequence (all appended tokens, quantized or not)
 *   layers: num_layers entries, read during kvq_create() only. */
typedef struct {
  int32_t num_layers;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t group_size;
  int32_t max_tokens;
  const kvq_layer_cfg* layers;
} kvq_config;

typedef struct kvq_handle kvq_handle;

/* Device layout of one layer, for tests and for callers that snapshot the
 * cache.  All pointers are device pointers into the buffer given to
 * kvq_create(); counts are the host's view after the calls issued so far.
 *
 * Per (batch b, kv head h) "unit" u = b * num_kv_heads + h:
 *   records + u * unit_record_stride is a sequence of group records, one per
 *   quantized key group (group j covers tokens [j*G, (j+1)*G)), each
 *   record_bytes long:
 *     [K codes: G rows x k_words u32][V codes: G rows x v_words u32]
 *     [K scale: head_dim f16][K zero: head_dim f16]   (per-channel keys), or
 *     [K (scale, zero): G pairs of f16]               (per-token keys)
 *     [V (scale, zero): G pairs of f16]
 *   With 2-, 4- or 8-bit keys each per-channel key row is stored in 8-channel
 *   chunks, chunk j of each channel quarter side by side: position 4j + t
 *   holds the channels of chunk t*head_dim/32 + j (head_dim 64: chunks
 *   0 2 4 6 1 3 5 7); 3-bit keys keep channel order.
 *   A code row is one token's head_dim codes, least significant field first:
 *   for b in {2,4,8} field j of word w is channel w*32/b + j at bits [b*j, b*j+b);
 *   for b = 3 word w holds channels 11w .. 11w+10, fields 0..9 3-bit at bit 3j
 *   and field 10 2-bit at bits 30..31.  Packed word w of token row t (t counted
 *   inside the record) is stored at index w XOR x: key rows of 32 words:
 *   x = 4 on odd t; value rows of 16 words: x = 8 when t & 2; value rows of 32
 *   words: x = 8 * (t & 3); all other rows x = 0.
 *   residual_k + u * residual_stride (and residual_v likewise) is a ring of
 *   `residual` slots of head_dim fp16 holding the window tokens
 *   [quantized_tokens, tokens); token i sits in slot i % residual, and
 *   the 16-byte chunk c of a slot s is stored at chunk position c ^ (s & 7). */
typedef struct {
  int32_t k_bits, v_bits, residual, group_size, head_dim;
  int32_t k_words, v_words;          /* u32 words per code row                */
  int32_t key_mode;                  /* KVQ_KEY_PER_CHANNEL or _PER_TOKEN     */
  int64_t record_bytes;
  int64_t unit_record_stride;        /* bytes between units' record arrays    */
  int64_t residual_stride;           /* bytes between units' rings            */
  int64_t tokens;                    /* tokens appended so far                */
  int64_t quantized_tokens;          /* tokens held as quantized groups       */
  int64_t residual_tokens;           /* tokens held in the FP16 ring          */
  const void* records;
  const void* residual_k;
  const void* residual_v;
  int32_t window_bound;              /* current window bound C (<= residual) */
  int32_t rpc_percent;               /* the layer's RPC ratio (0: static)     */
} kvq_layer_view;

/* Bytes of device memory the caller must provide for `cfg` (0 if cfg is
 * invalid).  Includes every layer's cache sized for max_tokens, per-layer
 * state and the decode workspace. */
size_t kvq_cache_bytes(const kvq_config* cfg);

/* Validate `cfg`, lay the caches out in `dev_buf` (device memory, 256-byte
 * aligned, `bytes` >= kvq_cache_bytes(cfg)), zero it, and select the kernel
 * instantiations for every layer's (k_bits, v_bits, head_dim, heads-per-kv)
 * once, so that later calls dispatch with a table lookup.  Writes a new handle
 * to *out.  Synchronizes the device once (the zeroing). */
kvq_status kvq_create(const kvq_config* cfg, void* dev_buf, size_t bytes, kvq_handle** out);

/* Append n_tokens (>= 0) new tokens to `layer`, oldest first.
 * K, V: device, fp16, [batch][num_kv_heads][n_tokens][head_dim] contiguous,
 * read-only, caller-owned.  New tokens enter the FP16 window; while the
 * window holds the layer's bound (`residual`, or less after an RPC shrink,
 * see kvq_layer_cfg) or more tokens, the oldest group_size tokens are
 * quantized (keys per channel, values per token), packed and stored as the
 * next group record, all in the launched kernels.  Used for prefill
 * (n_tokens = prompt length) and for decode (n_tokens = 1).
 * KVQ_ERR_CAPACITY if tokens + n_tokens > max_tokens. */
kvq_status kvq_append(kvq_handle* h, int layer, const void* K, const void* V, int n_tokens,
                      void* stream);

/* Decode attention of one query token per sequence over everything appended
 * to `layer` so far.
 * q: device fp16 [batch][num_q_heads][head_dim]; query head j reads kv head
 *    j / (num_q_heads / num_kv_heads).
 * out: device fp32 [batch][num_q_heads][head_dim], written entirely.
 * Scores are scaled by 1/sqrt(head_dim).  KVQ_ERR_STATE if the layer is empty.
 * The kernel is launched as a programmatic dependent of the previous kernel on
 * the stream: its CTAs may start while that kernel drains, but each waits for
 * it to complete before its first read, so stream order holds as usual. */
kvq_status kvq_decode_attn(kvq_handle* h, int layer, const void* q, float* out, void* stream);

/* Causal attention of the queries of the n_queries newest tokens over `layer`
 * as it stands: prefill or chunked-prefill attention over the quantized cache
 * (KVTuner, section A2, calibration design: prefill runs over the dequantized
 * cache; the attention is its A3 equation).  Call after appending the chunk.
 * With T tokens appended, query i (0 <= i < n_queries) belongs to the token at
 * position T - n_queries + i and attends the tokens at positions
 * 0 .. T - n_queries + i: quantized groups dequantized (code * s + z), window
 * tokens as stored.  Scores are scaled by 1/sqrt(head_dim).
 * q: device fp16 [batch][num_q_heads][n_queries][head_dim], 16-byte aligned;
 *    query head j reads kv head j / (num_q_heads / num_kv_heads).
 * out: device fp32 [batch][num_q_heads][n_queries][head_dim], written entirely.
 * workspace: caller-owned device scratch of at least
 *    kvq_chunk_workspace_bytes(h) bytes, 16-byte aligned; the layer's tiles are
 *    dequantized into it once, then read by the tensor-core kernel.  Its
 *    contents are overwritten; a call must not share it with another in flight.
 * KVQ_ERR_ARG if n_queries < 1 or > tokens appended; KVQ_ERR_STATE if the layer
 * is empty; KVQ_ERR_CAPACITY if the workspace is too small;
 * KVQ_ERR_UNSUPPORTED if batch * num_kv_heads > 65535.  Runs on the tensor
 * cores (tcgen05). */
kvq_status kvq_chunk_attn(kvq_handle* h, int layer, const void* q, int n_queries, float* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Bytes of the workspace kvq_chunk_attn needs for any layer of `h` (its
 * dequantized tiles of every (batch, kv head) at max_tokens).  0 if h is null. */
size_t kvq_chunk_workspace_bytes(const kvq_handle* h);

/* One decode step over every layer: for l = 0 .. num_layers-1,
 * kvq_append(l, K[l], V[l], 1) then kvq_decode_attn(l, q[l], out[l]).
 * K, V, q, out are host arrays of num_layers device pointers, with the shapes
 * above (n_tokens = 1).  The launches of a step do not depend on the cache
 * state, so after the first call with a given set of pointers the step is
 * replayed from a CUDA graph the handle keeps (it is re-captured when the
 * pointers change).  Inside the graph the appends run on a forked stream:
 * decode l waits for append l (and for decode l-1), so later layers' appends
 * overlap earlier layers' decodes.  Decode l is a programmatic dependent of
 * decode l-1: it stages its first items of layer l's cache (which decode l-1
 * does not write) while decode l-1 drains, and reads q[l] and writes out[l]
 * only after it.  KVQ_ERR_CAPACITY if any layer is full. */
kvq_status kvq_decode_step(kvq_handle* h, const void* const* K, const void* const* V,
                           const void* const* q, float* const* out, void* stream);

/* Size of the library's own device scratch for kvq_decode_attn_noalloc():
 * 4 MiB, a file-scope device array that every GPU which loads the library
 * keeps until the process exits. */
#define KVQ_NOALLOC_SCRATCH_BYTES (4u << 20)

/* kvq_decode_attn() for callers that may not allocate device memory at all.
 *
 * The papers have no counterpart to this entry point; it exists for callers
 * such as plugins hosted by another runtime that owns every device
 * allocation, or code on a latency path where cudaMalloc (which synchronises
 * the device) is not allowed.  Such a caller may hold a cache whose buffer it
 * cannot grow, and cannot hand the library extra workspace.
 *
 * Same arguments, result and errors as kvq_decode_attn(), except that the
 * split-merge workspace (per-split partial results and one arrival counter
 * per (batch, kv head) unit) comes from the library's static device array of
 * KVQ_NOALLOC_SCRATCH_BYTES instead of the handle's buffer, and nothing is
 * allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Needs align256(units * 4) + (grid + units) * gqa * (head_dim + 2) * 4
 *     bytes, where units = batch * num_kv_heads and grid is the layer's
 *     launch width (at most 1024 CTAs); a layer needing more returns
 *     KVQ_ERR_CAPACITY and launches nothing.
 *   - The current device must be the one that was current at kvq_create()
 *     (the device holding the handle's buffer); otherwise KVQ_ERR_ARG and
 *     nothing is launched.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress and keeps it; make that first call before any
 *     stream capture.  KVQ_ERR_CUDA if the lookup fails.
 *   - Each call clears the counters on `stream` (an asynchronous memset of
 *     units * 4 bytes) before it launches the kernel.
 *   - Every call on a device shares the one array: calls that overlap on the
 *     GPU (other streams, or other handles, without ordering between them)
 *     race on it and give wrong results.  Order them on one stream. */
kvq_status kvq_decode_attn_noalloc(kvq_handle* h, int layer, const void* q, float* out, void* stream);

/* Describe `layer` (see kvq_layer_view). */
kvq_status kvq_layer_view_get(const kvq_handle* h, int layer, kvq_layer_view* v);

/* f_m: mean over layers of (k_bits + v_bits) / 2 (KVTuner section A2). */
double kvq_equivalent_bits(const kvq_handle* h);

/* Algorithmic bytes one kvq_decode_attn(layer) call reads for the current
 * state (packed codes, scales/zeros, FP16 window, q) and writes (out). */
int64_t kvq_decode_bytes(const kvq_handle* h, int layer);

/* Reads the device error word (a bounded wait that gave up, or an internal
 * consistency check), clearing it.  Synchronizes `stream`.  0 means none. */
kvq_status kvq_device_error(kvq_handle* h, int32_t* code, void* stream);

/* Failure-detection self-test of the device-side waits.  Launches one warp
 * that waits on an mbarrier nothing ever completes, with a short bound (4096
 * tries), as every wait in the library is bounded.  The wait must give up,
 * record the timeout in the error word and return, with the CUDA context
 * still usable.  KVQ_OK if exactly that happened (the word is read and
 * cleared), KVQ_ERR_STATE if the timeout was not reported.  Synchronizes
 * `stream`; changes nothing else. */
kvq_status kvq_selftest_bounded_wait(kvq_handle* h, void* stream);

/* Snapshots of the streaming state, to rewind a cache to an earlier point
 * (re-running a window of decode steps, or dropping tokens decoded after the
 * snapshot).  A snapshot holds every layer's token counters (appended tokens,
 * quantized tokens, window bound, of every (batch, kv head) unit) and its FP16
 * residual window ring; it does not hold the quantized groups.  That is enough:
 * an append only writes groups at or past the quantized-token count it starts
 * from, and attention reads only groups below the current count, so a group
 * the snapshot does not hold is written again before anything reads it
 * (the cache is the groups quantized so far plus the FP16 window: KIVI notes
 * section 6.2, KVmix 关键设计 3).
 *
 * kvq_state_bytes: bytes of a snapshot of `h` (0 if h is null).
 *
 * kvq_state_save: copies the state into `dst`, a caller-owned device buffer of
 * kvq_state_bytes(h) bytes, 16-byte aligned, on `stream` after the work already
 * queued there (plain device-to-device copies, one per layer plus one for the
 * counters).  KVQ_ERR_ARG if h or dst is null, KVQ_ERR_ALIGN if dst is not
 * 16-byte aligned.
 *
 * kvq_state_restore: makes `src` (a snapshot saved from `h`, or from a handle
 * created with the same configuration) the cache's state.  It first reads the
 * snapshot's counters to the host (synchronizing `stream`) and checks that they
 * describe a state the cache can be in: every unit of a layer agrees, the
 * quantized count is a multiple of G and at most the appended count, which is
 * at most max_tokens, the window holds fewer tokens than its bound, and the
 * bound is a multiple of G between G and R_l (R_l itself on a static window).
 * KVQ_ERR_STATE if not, and nothing changes.  Otherwise the copies back are
 * queued on `stream` and the host mirror is set from the snapshot.  A captured
 * decode step stays valid (its launches read the state from the device). */
size_t kvq_state_bytes(const kvq_handle* h);
kvq_status kvq_state_save(kvq_handle* h, void* dst, void* stream);
kvq_status kvq_state_restore(kvq_handle* h, const void* src, void* stream);

/* Release the handle (host memory and any captured graph).  The device buffer
 * stays the caller's. */
kvq_status kvq_destroy(kvq_handle* h);

const char* kvq_status_string(kvq_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
