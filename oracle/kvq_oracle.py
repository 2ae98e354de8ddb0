"""Oracle for layer-wise mixed-precision KV-cache quantization and decode attention.

TEST INFRASTRUCTURE ONLY.  This is the plain, slow CPU statement of what the
CUDA path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import it; the library itself never does.  It
shares no code with the CUDA path: it reads fp16 inputs and produces the packed
cache bytes and fp64 attention outputs from the definitions below.

Sources (web pages, cited by title and section):

* [KVTuner] "KVTuner: Sensitivity-Aware Layer-Wise Mixed-Precision KV Cache
  Quantization for Efficient and Nearly Lossless LLM Inference", section A3
  (attention equation; quantizer Q(X) = round((X - z)/s), z = min X,
  s = (max X - min X)/(2^B - 1); error metrics e_k, e_v, e_a, e_o) and section
  A2 (f_m, the mean equivalent bit width; KxVy pairs per layer).
* [KVmix] "KVmix: Gradient-Based Layer Importance-Aware Mixed-Precision
  Quantization for KV Cache", 关键设计 2 (keys per channel, values per token,
  s = (max - min)/q_max, codes packed into int32, 3-bit words of ten 3-bit and
  one 2-bit field) and 关键设计 3 (per-layer full-precision recent window).
* [KIVI notes] "LLM 量化精读笔记 · 08 KV Cache 量化：KIVI 与误差累积", section
  2.1 (KV bytes formula), 2.2 (Llama-2-70B example), 6.1-6.2 (per-channel
  keys over token segments, per-token values, FP16 buffer of recent tokens,
  streaming quantization), exercise 1 (64 layers x 4 kv heads x d128 x 64K).

Readings taken where the pages leave a step open (each also listed in the
design notes):

* "round" is round-half-to-even (``rint``), after the fp32 IEEE subtraction
  ``x - min`` and division by the *stored* fp16 scale; s = 0 gives code 0.
* the scale is computed in fp32 as (max - min)/(2^b - 1) and stored as fp16
  (round to nearest even); the zero is min, exact in fp16.
* 3-bit: 11 channels per 32-bit word, fields 0..9 are 3-bit at bit 3j and field
  10 is 2-bit at bits 30..31; field 10 is coded with s2 = (s * 7) / 3 (fp32) and
  clamped to 0..3, and dequantized with s2.
* attention scale is 1/sqrt(head_dim); the new token is appended before the
  query attends (K = concat(K_{:i-1}, k_i)).
* streaming: tokens enter an FP16 residual window of R_l tokens; whenever the
  window holds R_l or more tokens the oldest G are quantized as one key group
  (keys per channel over those G tokens, values per token).
* KVmix's dynamic window (RPC: num_RPC = floor(r x current_RPC), shrinking as
  decoding proceeds): a layer with an RPC ratio of p percent keeps a window
  bound C, first R_l (the prefill's p% of the prompt).  When a single-token
  (decode) append brings the window to C or more tokens, the bound becomes
  C' = G * max(1, floor(p * C / (100 * G))) -- the ratio applied to the FP16
  tokens held, rounded down to whole key groups and never below one group --
  and then the oldest G are quantized while the window holds C' or more.
  Multi-token appends (prefill, chunks) keep the current bound.  The ring
  keeps its R_l slots (token i in slot i mod R_l), since C <= R_l.

Layout of the quantized cache (mirrored by the CUDA path):

* codes are packed LSB first: in a b-bit word (b in 2, 4, 8) field j holds the
  code of channel (word * 32/b + j) at bits [b*j, b*j + b); a token's d codes
  are contiguous ("token-major" rows of d*b/32 words, or ceil(d/11) words for
  3 bits);
* per (batch, kv head) the cache is a sequence of group records, one per key
  group of G tokens:
  ``[K codes G x WK u32][V codes G x WV u32][K scale d f16][K zero d f16]
  [V (scale, zero) G pairs of f16]`` (each token's value scale and zero adjacent);
* the residual window is a ring of R_l slots; token i (absolute position) sits
  in slot i mod R_l; K rows then V rows, d fp16 each.
"""

from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np

F16 = np.float16
F32 = np.float32

BITS_ALLOWED = (2, 3, 4, 8)


# --------------------------------------------------------------------------
# Memory formulas
# --------------------------------------------------------------------------

def kv_cache_bytes(n_layers: int, n_kv_heads: int, head_dim: int, seq_len: int,
                   bytes_per_elem: float) -> float:
    """K and V cache bytes: 2 * layers * kv heads * head_dim * tokens * bytes
    ([KIVI notes] section 2.1)."""
    return 2 * n_layers * n_kv_heads * head_dim * seq_len * bytes_per_elem


def equivalent_bits(pairs: Sequence[Tuple[int, int]]) -> float:
    """f_m: mean equivalent bit width over layers, (k_bits + v_bits)/2 per
    layer ([KVTuner] section A2, problem formulation)."""
    return sum((kb + vb) / 2.0 for kb, vb in pairs) / len(pairs)


# --------------------------------------------------------------------------
# Asymmetric uniform quantizer ([KVTuner] A3; [KVmix] 关键设计 2)
# --------------------------------------------------------------------------

def asym_scale(mn: np.ndarray, mx: np.ndarray, bits: int) -> np.ndarray:
    """fp16 scale s = (max - min)/(2^b - 1), evaluated in fp32, stored fp16."""
    mn32 = np.asarray(mn, dtype=F16).astype(F32)
    mx32 = np.asarray(mx, dtype=F16).astype(F32)
    s32 = (mx32 - mn32) / F32(2 ** bits - 1)
    return s32.astype(F16)


def asym_codes(x: np.ndarray, mn: np.ndarray, s: np.ndarray, qmax: int) -> np.ndarray:
    """code = clamp(rint((x - min)/s), 0, qmax) in fp32; s == 0 gives 0.

    ``s`` is the fp32 value of the stored scale (or the derived 2-bit field
    scale for 3-bit words)."""
    x32 = np.asarray(x, dtype=F16).astype(F32)
    mn32 = np.asarray(mn, dtype=F16).astype(F32)
    s32 = np.asarray(s, dtype=F32)
    diff = x32 - mn32
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = diff / s32
    q = np.rint(quot)
    q = np.where(s32 == F32(0), F32(0), q)
    q = np.clip(q, F32(0), F32(qmax))
    return q.astype(np.uint8)


def slot10_scale(s16: np.ndarray) -> np.ndarray:
    """Scale of the 2-bit field of a 3-bit word: (s * 7) / 3 in fp32."""
    return (np.asarray(s16, dtype=F16).astype(F32) * F32(7.0)) / F32(3.0)


def is_slot10(d: int) -> np.ndarray:
    """Channels that land in the 2-bit field of an 11-field 3-bit word."""
    c = np.arange(d)
    return (c % 11) == 10


def quantize_keys_group(k: np.ndarray, bits: int):
    """Per-channel key quantization over one group of G tokens.

    k: [G, d] fp16.  Returns (codes [G, d] u8, scale [d] f16, zero [d] f16).
    One (scale, zero) per channel over the group's tokens ([KIVI notes] 6.1,
    6.2; [KVmix] 关键设计 2)."""
    k = np.asarray(k, dtype=F16)
    mn = k.min(axis=0)
    mx = k.max(axis=0)
    s16 = asym_scale(mn, mx, bits)
    if bits == 3:
        d = k.shape[1]
        two = is_slot10(d)
        s_eff = np.where(two, slot10_scale(s16), s16.astype(F32)).astype(F32)
        codes = np.empty(k.shape, dtype=np.uint8)
        codes[:, ~two] = asym_codes(k[:, ~two], mn[~two], s_eff[~two], 7)
        codes[:, two] = asym_codes(k[:, two], mn[two], s_eff[two], 3)
    else:
        codes = asym_codes(k, mn[None, :], s16.astype(F32)[None, :], 2 ** bits - 1)
    return codes, s16, mn.astype(F16)


def quantize_values_tokens(v: np.ndarray, bits: int):
    """Per-token value quantization.

    v: [n, d] fp16.  Returns (codes [n, d] u8, scale [n] f16, zero [n] f16).
    One (scale, zero) per token over its d channels ([KIVI notes] 6.1, 6.2;
    [KVmix] 关键设计 2)."""
    v = np.asarray(v, dtype=F16)
    mn = v.min(axis=1)
    mx = v.max(axis=1)
    s16 = asym_scale(mn, mx, bits)
    if bits == 3:
        d = v.shape[1]
        two = is_slot10(d)
        codes = np.empty(v.shape, dtype=np.uint8)
        s3 = s16.astype(F32)[:, None]
        s2 = slot10_scale(s16)[:, None]
        codes[:, ~two] = asym_codes(v[:, ~two], mn[:, None], s3, 7)
        codes[:, two] = asym_codes(v[:, two], mn[:, None], s2, 3)
    else:
        codes = asym_codes(v, mn[:, None], s16.astype(F32)[:, None], 2 ** bits - 1)
    return codes, s16, mn.astype(F16)


# --------------------------------------------------------------------------
# int32 packing ([KVmix] 关键设计 2)
# --------------------------------------------------------------------------

def words_per_row(d: int, bits: int) -> int:
    if bits == 3:
        return (d + 10) // 11
    return d * bits // 32


def pack_rows(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes [n, d] u8 -> words [n, WK] u32, LSB first."""
    codes = np.asarray(codes, dtype=np.uint32)
    n, d = codes.shape
    nw = words_per_row(d, bits)
    out = np.zeros((n, nw), dtype=np.uint32)
    if bits == 3:
        for c in range(d):
            w, j = divmod(c, 11)
            shift = 30 if j == 10 else 3 * j
            out[:, w] |= codes[:, c] << np.uint32(shift)
    else:
        per = 32 // bits
        for c in range(d):
            w, j = divmod(c, per)
            out[:, w] |= codes[:, c] << np.uint32(bits * j)
    return out


def unpack_rows(words: np.ndarray, bits: int, d: int) -> np.ndarray:
    """words [n, WK] u32 -> codes [n, d] u8 (inverse of pack_rows)."""
    words = np.asarray(words, dtype=np.uint32)
    n = words.shape[0]
    out = np.zeros((n, d), dtype=np.uint8)
    if bits == 3:
        for c in range(d):
            w, j = divmod(c, 11)
            if j == 10:
                out[:, c] = (words[:, w] >> np.uint32(30)) & np.uint32(3)
            else:
                out[:, c] = (words[:, w] >> np.uint32(3 * j)) & np.uint32(7)
    else:
        per = 32 // bits
        mask = np.uint32(2 ** bits - 1)
        for c in range(d):
            w, j = divmod(c, per)
            out[:, c] = (words[:, w] >> np.uint32(bits * j)) & mask
    return out


# --------------------------------------------------------------------------
# Dequantization (fp64)
# --------------------------------------------------------------------------

def dequant_keys(codes: np.ndarray, s16: np.ndarray, z16: np.ndarray, bits: int) -> np.ndarray:
    """x_hat = code * s + z per channel, in fp64 ([KVTuner] A3)."""
    s = np.asarray(s16, dtype=F16).astype(np.float64)
    if bits == 3:
        two = is_slot10(codes.shape[1])
        s = np.where(two, slot10_scale(s16).astype(np.float64), s)
    return codes.astype(np.float64) * s[None, :] + np.asarray(z16, dtype=F16).astype(np.float64)[None, :]


def dequant_values(codes: np.ndarray, s16: np.ndarray, z16: np.ndarray, bits: int) -> np.ndarray:
    s = np.asarray(s16, dtype=F16).astype(np.float64)[:, None]
    z = np.asarray(z16, dtype=F16).astype(np.float64)[:, None]
    if bits == 3:
        two = is_slot10(codes.shape[1])[None, :]
        s2 = slot10_scale(s16).astype(np.float64)[:, None]
        s = np.where(two, s2, s)
    return codes.astype(np.float64) * s + z


# --------------------------------------------------------------------------
# Attention (fp64, two pass) ([KVTuner] A3 equation)
# --------------------------------------------------------------------------

def attention_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """a = softmax(q K^T / sqrt(d)), o = a V for one query head.

    q [d], k [T, d], v [T, d] (any float) -> o [d] fp64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d = q.shape[0]
    scores = (k * q[None, :]).sum(axis=1) / math.sqrt(d)
    m = scores.max()
    p = np.exp(scores - m)
    a = p / p.sum()
    return (a[:, None] * v).sum(axis=0)


def gqa_attention_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """q [Hq, d], k/v [Hkv, T, d] -> out [Hq, d]; query head h reads kv head
    h // (Hq / Hkv)."""
    hq = q.shape[0]
    hkv = k.shape[0]
    rep = hq // hkv
    out = np.zeros((hq, q.shape[1]), dtype=np.float64)
    for h in range(hq):
        out[h] = attention_fp64(q[h], k[h // rep], v[h // rep])
    return out


# --------------------------------------------------------------------------
# Streaming state machine ([KIVI notes] 6.2; [KVmix] 关键设计 3)
# --------------------------------------------------------------------------

def shrink_bound(bound: int, rpc_percent: int, group: int) -> int:
    """KVmix 关键设计 3: num_RPC = floor(r x current_RPC) with r the layer's RPC
    ratio (percent here) and current_RPC the FP16 tokens held (the bound C when
    a decode step reaches it), rounded down to whole key groups, at least one."""
    return group * max(1, (rpc_percent * bound) // (100 * group))


def flush_state(total: int, residual: int, group: int) -> Tuple[int, int]:
    """(quantized tokens, residual tokens) after ``total`` appended tokens,
    found by replaying the rule token by token: append, then while the
    window holds >= R tokens quantize the oldest G."""
    n_q, r = 0, 0
    for _ in range(total):
        r += 1
        while r >= residual:
            n_q += group
            r -= group
    return n_q, r


# Key quantization modes ([KVTuner] A3 and A4: the KIVI mode and the
# per-token-asym mode, chosen per layer together with its precision pair)
KEY_PER_CHANNEL = 0   # keys per channel over the G tokens of a group (KIVI)
KEY_PER_TOKEN = 1     # keys per token over their d channels, like values


def key_scale_chunk_order(d: int) -> np.ndarray:
    """Storage order of the per-channel key scale row and zero row of a record
    with 2-, 4- or 8-bit keys (3-bit keys keep the natural channel order).

    The pages fix the values (one fp16 scale and zero per channel and group), not
    where a record keeps them; this is the library's storage decision.  Split the
    d channels into chunks of 8 and the chunks into 4 equal quarters; the row
    stores chunk j of every quarter together: position 4*j + t holds chunk
    t*(d/32) + j.  Returns, for each stored position, the natural chunk index."""
    per_quarter = d // 32
    order = np.empty(d // 8, dtype=np.int64)
    for t in range(4):
        for j in range(per_quarter):
            order[4 * j + t] = t * per_quarter + j
    return order


def key_scale_row_store(row: np.ndarray) -> np.ndarray:
    """A length-d per-channel row (natural channel order) in record storage order."""
    d = row.shape[0]
    chunks = row.reshape(d // 8, 8)
    return chunks[key_scale_chunk_order(d)].reshape(d)


def key_scale_row_load(stored: np.ndarray) -> np.ndarray:
    """Inverse of key_scale_row_store: back to natural channel order."""
    d = stored.shape[0]
    out = np.empty((d // 8, 8), dtype=stored.dtype)
    out[key_scale_chunk_order(d)] = stored.reshape(d // 8, 8)
    return out.reshape(d)


def code_row_word_xor(words_per_token: int, is_key: bool, t: int) -> int:
    """Where token row t (0-based inside its record) keeps its packed words.

    Like the scale rows, this is the library's storage decision; the pages fix
    the packing inside a word only.  Word w of the row is stored at index
    w XOR (the value returned):
      keys with 32 words a row (8-bit, d = 128): 4 on odd rows, else 0;
      values with 16 words a row: 8 when bit 1 of t is set, else 0;
      values with 32 words a row: 8 * (t mod 4);
      every other row is stored as packed (0)."""
    if is_key:
        return 4 * (t % 2) if words_per_token == 32 else 0
    if words_per_token == 16:
        return 8 if (t // 2) % 2 == 1 else 0
    if words_per_token == 32:
        return 8 * (t % 4)
    return 0


def code_rows_store(words: np.ndarray, is_key: bool) -> np.ndarray:
    """Packed rows [G, W] (row t = token t of the record) in storage order."""
    n, w = words.shape
    out = np.empty_like(words)
    for t in range(n):
        x = code_row_word_xor(w, is_key, t)
        for i in range(w):
            out[t, i ^ x] = words[t, i]
    return out


def code_rows_load(stored: np.ndarray, is_key: bool) -> np.ndarray:
    """Inverse of code_rows_store."""
    n, w = stored.shape
    out = np.empty_like(stored)
    for t in range(n):
        x = code_row_word_xor(w, is_key, t)
        for i in range(w):
            out[t, i] = stored[t, i ^ x]
    return out


def record_layout(d: int, group: int, k_bits: int, v_bits: int, key_mode: int = KEY_PER_CHANNEL) -> Dict[str, int]:
    """Byte offsets inside one group record.

    Per-channel keys: [K codes][V codes][K scale d][K zero d][V (scale, zero) G],
    the two d-long rows in key_scale_chunk_order (2-, 4-, 8-bit keys; channel
    order for 3-bit keys); code rows in the word order of code_row_word_xor.
    Per-token keys:   [K codes][V codes][K (scale, zero) G][V (scale, zero) G]."""
    wk = words_per_row(d, k_bits)
    wv = words_per_row(d, v_bits)
    off = {}
    off["k_codes"] = 0
    off["v_codes"] = off["k_codes"] + 4 * group * wk
    off["k_scale"] = off["v_codes"] + 4 * group * wv
    if key_mode == KEY_PER_TOKEN:
        off["k_zero"] = off["k_scale"]            # interleaved with the scales
        off["v_scale"] = off["k_scale"] + 4 * group
    else:
        off["k_zero"] = off["k_scale"] + 2 * d
        off["v_scale"] = off["k_zero"] + 2 * d    # (scale, zero) pairs, one per token
    off["bytes"] = off["v_scale"] + 4 * group
    off["wk"] = wk
    off["wv"] = wv
    return off


def build_group_record(k_grp: np.ndarray, v_grp: np.ndarray, k_bits: int, v_bits: int,
                       key_mode: int = KEY_PER_CHANNEL) -> bytes:
    """Quantize one key group (k_grp, v_grp: [G, d] fp16) and lay out its record."""
    vc, vs, vz = quantize_values_tokens(v_grp, v_bits)
    vsz = np.stack([vs.astype(F16), vz.astype(F16)], axis=1)  # [G, 2]
    if key_mode == KEY_PER_TOKEN:
        kc, ks, kz = quantize_values_tokens(k_grp, k_bits)
        kparts = [np.stack([ks.astype(F16), kz.astype(F16)], axis=1).tobytes()]
    else:
        kc, ks, kz = quantize_keys_group(k_grp, k_bits)
        ks, kz = ks.astype(F16), kz.astype(F16)
        if k_bits != 3:
            ks, kz = key_scale_row_store(ks), key_scale_row_store(kz)
        kparts = [ks.tobytes(), kz.tobytes()]
    parts = [code_rows_store(pack_rows(kc, k_bits), True).tobytes(),
             code_rows_store(pack_rows(vc, v_bits), False).tobytes(), *kparts, vsz.tobytes()]
    return b"".join(parts)


def parse_group_record(rec: bytes, d: int, group: int, k_bits: int, v_bits: int,
                       key_mode: int = KEY_PER_CHANNEL):
    """Inverse of build_group_record's layout: returns dequantized K, V [G, d] fp64."""
    lay = record_layout(d, group, k_bits, v_bits, key_mode)
    buf = np.frombuffer(rec, dtype=np.uint8)
    kw = code_rows_load(buf[lay["k_codes"]:lay["v_codes"]].view(np.uint32).reshape(group, lay["wk"]), True)
    vw = code_rows_load(buf[lay["v_codes"]:lay["k_scale"]].view(np.uint32).reshape(group, lay["wv"]), False)
    vsz = buf[lay["v_scale"]:lay["bytes"]].view(F16).reshape(group, 2)
    vs, vz = vsz[:, 0], vsz[:, 1]
    if key_mode == KEY_PER_TOKEN:
        ksz = buf[lay["k_scale"]:lay["v_scale"]].view(F16).reshape(group, 2)
        k_hat = dequant_values(unpack_rows(kw, k_bits, d), ksz[:, 0], ksz[:, 1], k_bits)
    else:
        ks = buf[lay["k_scale"]:lay["k_zero"]].view(F16)
        kz = buf[lay["k_zero"]:lay["v_scale"]].view(F16)
        if k_bits != 3:
            ks, kz = key_scale_row_load(ks), key_scale_row_load(kz)
        k_hat = dequant_keys(unpack_rows(kw, k_bits, d), ks, kz, k_bits)
    v_hat = dequant_values(unpack_rows(vw, v_bits, d), vs, vz, v_bits)
    return k_hat, v_hat


class OracleLayerCache:
    """One layer's quantized cache for B x Hkv independent (batch, kv head)
    units, fed in token order."""

    def __init__(self, batch: int, n_kv_heads: int, head_dim: int, group: int,
                 k_bits: int, v_bits: int, residual: int, key_mode: int = KEY_PER_CHANNEL,
                 rpc_percent: int = 0):
        if residual < group:
            raise ValueError("residual window must hold at least one key group")
        if not 0 <= rpc_percent <= 100:
            raise ValueError("RPC ratio is a percentage")
        self.B, self.H, self.d, self.G = batch, n_kv_heads, head_dim, group
        self.kb, self.vb, self.R = k_bits, v_bits, residual  # R: ring slots, the first bound
        self.key_mode = key_mode
        self.rpc = rpc_percent  # 0: static window of R tokens
        self.bound = residual   # the window bound C
        self.total = 0
        self.n_q = 0
        # per unit: list of group records; pending fp16 tokens (oldest first)
        self.records: List[List[bytes]] = [[] for _ in range(batch * n_kv_heads)]
        self.pend_k = np.zeros((batch * n_kv_heads, 0, head_dim), dtype=F16)
        self.pend_v = np.zeros((batch * n_kv_heads, 0, head_dim), dtype=F16)

    def append(self, k: np.ndarray, v: np.ndarray) -> None:
        """k, v: [B, Hkv, n, d] fp16, oldest token first."""
        k = np.asarray(k, dtype=F16).reshape(self.B * self.H, -1, self.d)
        v = np.asarray(v, dtype=F16).reshape(self.B * self.H, -1, self.d)
        n = k.shape[1]
        self.pend_k = np.concatenate([self.pend_k, k], axis=1)
        self.pend_v = np.concatenate([self.pend_v, v], axis=1)
        self.total += n
        if n == 1 and self.rpc > 0 and self.pend_k.shape[1] >= self.bound:
            self.bound = shrink_bound(self.bound, self.rpc, self.G)  # a decode step reached the bound
        while self.pend_k.shape[1] >= self.bound:
            for u in range(self.B * self.H):
                self.records[u].append(build_group_record(
                    self.pend_k[u, : self.G], self.pend_v[u, : self.G], self.kb, self.vb, self.key_mode))
            self.pend_k = self.pend_k[:, self.G:]
            self.pend_v = self.pend_v[:, self.G:]
            self.n_q += self.G

    @property
    def r(self) -> int:
        return self.pend_k.shape[1]

    def record_bytes(self) -> int:
        return record_layout(self.d, self.G, self.kb, self.vb, self.key_mode)["bytes"]

    def unit_records(self, u: int) -> bytes:
        return b"".join(self.records[u])

    def residual_ring(self, u: int) -> Tuple[np.ndarray, np.ndarray]:
        """Ring contents [R, d] fp16 for K and V: token i in slot i mod R; slots
        not holding a live residual token are left zero."""
        rk = np.zeros((self.R, self.d), dtype=F16)
        rv = np.zeros((self.R, self.d), dtype=F16)
        for i in range(self.r):
            pos = self.n_q + i
            rk[pos % self.R] = self.pend_k[u, i]
            rv[pos % self.R] = self.pend_v[u, i]
        return rk, rv

    def live_ring_slots(self) -> np.ndarray:
        return np.array([(self.n_q + i) % self.R for i in range(self.r)], dtype=np.int64)

    def dequantized(self, u: int) -> Tuple[np.ndarray, np.ndarray]:
        """All appended tokens of unit u as fp64 [T, d] (quantized groups
        dequantized, residual tokens exact)."""
        ks, vs = [], []
        for rec in self.records[u]:
            kh, vh = parse_group_record(rec, self.d, self.G, self.kb, self.vb, self.key_mode)
            ks.append(kh)
            vs.append(vh)
        ks.append(self.pend_k[u].astype(np.float64))
        vs.append(self.pend_v[u].astype(np.float64))
        return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)

    def attend(self, q: np.ndarray, units: Sequence[int] = None) -> np.ndarray:
        """q: [B, Hq, d] fp16 -> out [B, Hq, d] fp64 (rows of units not listed
        stay NaN)."""
        q = np.asarray(q, dtype=F16)
        B, Hq, d = q.shape
        rep = Hq // self.H
        out = np.full((B, Hq, d), np.nan)
        if units is None:
            units = range(self.B * self.H)
        for u in units:
            b, h = divmod(u, self.H)
            kh, vh = self.dequantized(u)
            for j in range(rep):
                out[b, h * rep + j] = attention_fp64(q[b, h * rep + j].astype(np.float64), kh, vh)
        return out


    def attend_chunk(self, q: np.ndarray, units: Sequence[int] = None) -> np.ndarray:
        """Causal attention of the n newest tokens' queries over the cache.

        q: [B, Hq, n, d] fp16, query i belonging to the token at position
        T - n + i (T = tokens appended so far).  It attends the tokens at
        positions 0 .. T - n + i of the cache as it stands: quantized groups
        dequantized, window tokens exact ([KVTuner] A2, calibration design: prefill
        attention over the dequantized cache; [KVTuner] A3 attention).
        Returns [B, Hq, n, d] fp64 (rows of units not listed stay NaN)."""
        q = np.asarray(q, dtype=F16)
        B, Hq, n, d = q.shape
        if not 1 <= n <= self.total:
            raise ValueError("chunk must hold between 1 and the appended tokens")
        rep = Hq // self.H
        out = np.full((B, Hq, n, d), np.nan)
        if units is None:
            units = range(self.B * self.H)
        for u in units:
            b, h = divmod(u, self.H)
            kh, vh = self.dequantized(u)
            for j in range(rep):
                for i in range(n):
                    last = self.total - n + i
                    out[b, h * rep + j, i] = attention_fp64(q[b, h * rep + j, i].astype(np.float64),
                                                            kh[: last + 1], vh[: last + 1])
        return out


# --------------------------------------------------------------------------
# Relative error metrics ([KVTuner] A3)
# --------------------------------------------------------------------------

def rel_error(x: np.ndarray, x_hat: np.ndarray) -> float:
    """mean(|X - X_hat| / |X|) over elements with X != 0."""
    x = np.asarray(x, dtype=np.float64)
    x_hat = np.asarray(x_hat, dtype=np.float64)
    nz = x != 0
    return float(np.mean(np.abs(x[nz] - x_hat[nz]) / np.abs(x[nz])))


def quantize_keys_per_token(k: np.ndarray, bits: int) -> np.ndarray:
    """Keys quantized per token (the per-token-asym mode), dequantized fp64;
    used only to compare error orderings."""
    codes, s, z = quantize_values_tokens(k, bits)
    return dequant_values(codes, s, z, bits)


# --------------------------------------------------------------------------
# Intra-layer Pareto pruning of precision pairs ([KVTuner] A2, two-stage
# search-space pruning, step 1: a layer's candidate KxVy pairs are cut to
# those not dominated in (equivalent bits, e_o))
# --------------------------------------------------------------------------

def pair_output_errors(k: np.ndarray, v: np.ndarray, queries: Sequence[np.ndarray],
                       pairs: Sequence[Tuple[int, int]], group: int, residual: int,
                       key_mode: int = KEY_PER_CHANNEL) -> Dict[Tuple[int, int], float]:
    """e_o of each pair on one layer's KV ([KVTuner] A3, quantization basics:
    e_o = mean(|o - o_hat| / |o|)).

    k, v: [B, Hkv, T, d] fp16; queries: [B, Hq, d] fp16 arrays.  o is fp64
    attention over the fp16 K and V; o_hat over the pair's quantized cache
    after appending all T tokens (window `residual`)."""
    k = np.asarray(k, dtype=F16)
    v = np.asarray(v, dtype=F16)
    B, H, T, d = k.shape
    out = {}
    for kb, vb in pairs:
        cache = OracleLayerCache(B, H, d, group, kb, vb, residual, key_mode)
        cache.append(k, v)
        o_all, oh_all = [], []
        for q in queries:
            q = np.asarray(q, dtype=F16)
            rep = q.shape[1] // H
            oh = cache.attend(q)
            for b in range(B):
                for h in range(q.shape[1]):
                    u = h // rep
                    o_all.append(attention_fp64(q[b, h].astype(np.float64), k[b, u].astype(np.float64),
                                                v[b, u].astype(np.float64)))
                    oh_all.append(oh[b, h])
        out[(kb, vb)] = rel_error(np.stack(o_all), np.stack(oh_all))
    return out


def pareto_front(errors: Dict[Tuple[int, int], float]) -> List[Tuple[int, int]]:
    """Pairs not dominated: no other pair has equivalent bits <= and e_o <=
    with at least one strictly smaller."""
    bits = {p: (p[0] + p[1]) / 2 for p in errors}
    keep = []
    for p in errors:
        dominated = any(bits[q] <= bits[p] and errors[q] <= errors[p] and (bits[q] < bits[p] or errors[q] < errors[p])
                        for q in errors if q != p)
        if not dominated:
            keep.append(p)
    return sorted(keep, key=lambda p: (bits[p], errors[p]))
