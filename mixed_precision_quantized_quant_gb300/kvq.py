"""Thin ctypes binding of libkvq.so (include/kvq.h).

Argument marshalling only: every step of quantization and attention runs in
the library's CUDA kernels.  PyTorch provides the device memory and streams.
The functions keep the C names; ``KVQCache`` bundles them for convenience.
There is no fallback: if the library is not built, loading it raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVQ_DEBUG_LIB=1 selects the debug build (device-side range checks of every
# computed access, reported through the error word)
LIB_PATH = os.path.join(_HERE, "libkvq_debug.so" if os.environ.get("KVQ_DEBUG_LIB") == "1" else "libkvq.so")

STATUS = {
    0: "KVQ_OK", 1: "KVQ_ERR_ARG", 2: "KVQ_ERR_BITS", 3: "KVQ_ERR_ALIGN", 4: "KVQ_ERR_CAPACITY",
    5: "KVQ_ERR_CUDA", 6: "KVQ_ERR_STATE", 7: "KVQ_ERR_UNSUPPORTED",
}

EXPORTS = (
    "kvq_cache_bytes", "kvq_create", "kvq_append", "kvq_decode_attn", "kvq_decode_step",
    "kvq_layer_view_get", "kvq_equivalent_bits", "kvq_decode_bytes", "kvq_device_error",
    "kvq_destroy", "kvq_status_string", "kvq_decode_attn_noalloc", "kvq_chunk_attn",
    "kvq_selftest_bounded_wait", "kvq_chunk_workspace_bytes", "kvq_state_bytes", "kvq_state_save",
    "kvq_state_restore",
)


class KVQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


KEY_PER_CHANNEL, KEY_PER_TOKEN = 0, 1


class LayerCfg(ctypes.Structure):
    _fields_ = [("k_bits", ctypes.c_uint8), ("v_bits", ctypes.c_uint8), ("key_mode", ctypes.c_uint8),
                ("rpc_percent", ctypes.c_uint8), ("residual", ctypes.c_int32)]


class Config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("layers", ctypes.POINTER(LayerCfg))]


class LayerView(ctypes.Structure):
    _fields_ = [("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32), ("residual", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("k_words", ctypes.c_int32), ("v_words", ctypes.c_int32), ("key_mode", ctypes.c_int32),
                ("record_bytes", ctypes.c_int64), ("unit_record_stride", ctypes.c_int64),
                ("residual_stride", ctypes.c_int64), ("tokens", ctypes.c_int64),
                ("quantized_tokens", ctypes.c_int64), ("residual_tokens", ctypes.c_int64),
                ("records", ctypes.c_void_p), ("residual_k", ctypes.c_void_p),
                ("residual_v", ctypes.c_void_p), ("window_bound", ctypes.c_int32),
                ("rpc_percent", ctypes.c_int32)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: build it with mixed_precision_quantized_quant_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.kvq_cache_bytes.argtypes = [ctypes.POINTER(Config)]
    L.kvq_cache_bytes.restype = ctypes.c_size_t
    L.kvq_create.argtypes = [ctypes.POINTER(Config), vp, ctypes.c_size_t, ctypes.POINTER(vp)]
    L.kvq_create.restype = ctypes.c_int
    L.kvq_append.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, vp]
    L.kvq_append.restype = ctypes.c_int
    L.kvq_decode_attn.argtypes = [vp, ctypes.c_int, vp, vp, vp]
    L.kvq_decode_attn.restype = ctypes.c_int
    L.kvq_decode_attn_noalloc.argtypes = [vp, ctypes.c_int, vp, vp, vp]
    L.kvq_decode_attn_noalloc.restype = ctypes.c_int
    L.kvq_chunk_attn.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]
    L.kvq_chunk_attn.restype = ctypes.c_int
    L.kvq_chunk_workspace_bytes.argtypes = [vp]
    L.kvq_chunk_workspace_bytes.restype = ctypes.c_size_t
    L.kvq_decode_step.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                  ctypes.POINTER(vp), vp]
    L.kvq_decode_step.restype = ctypes.c_int
    L.kvq_layer_view_get.argtypes = [vp, ctypes.c_int, ctypes.POINTER(LayerView)]
    L.kvq_layer_view_get.restype = ctypes.c_int
    L.kvq_equivalent_bits.argtypes = [vp]
    L.kvq_equivalent_bits.restype = ctypes.c_double
    L.kvq_decode_bytes.argtypes = [vp, ctypes.c_int]
    L.kvq_decode_bytes.restype = i64
    L.kvq_device_error.argtypes = [vp, ctypes.POINTER(i32), vp]
    L.kvq_device_error.restype = ctypes.c_int
    L.kvq_selftest_bounded_wait.argtypes = [vp, vp]
    L.kvq_selftest_bounded_wait.restype = ctypes.c_int
    L.kvq_state_bytes.argtypes = [vp]
    L.kvq_state_bytes.restype = ctypes.c_size_t
    L.kvq_state_save.argtypes = [vp, vp, vp]
    L.kvq_state_save.restype = ctypes.c_int
    L.kvq_state_restore.argtypes = [vp, vp, vp]
    L.kvq_state_restore.restype = ctypes.c_int
    L.kvq_destroy.argtypes = [vp]
    L.kvq_destroy.restype = ctypes.c_int
    L.kvq_status_string.argtypes = [ctypes.c_int]
    L.kvq_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(st: int, where: str) -> None:
    if st != 0:
        raise KVQError(st, where)


def make_config(layers: Sequence[Tuple[int, ...]], batch: int, num_q_heads: int, num_kv_heads: int,
                head_dim: int, group_size: int, max_tokens: int):
    """layers: (k_bits, v_bits, residual[, key_mode[, rpc_percent]]) per layer."""
    arr = (LayerCfg * len(layers))()
    for i, spec in enumerate(layers):
        kb, vb, r = spec[:3]
        km = spec[3] if len(spec) > 3 else KEY_PER_CHANNEL
        rpc = spec[4] if len(spec) > 4 else 0
        arr[i].k_bits, arr[i].v_bits, arr[i].key_mode, arr[i].rpc_percent, arr[i].residual = kb, vb, km, rpc, r
    cfg = Config(len(layers), batch, num_q_heads, num_kv_heads, head_dim, group_size, max_tokens,
                 ctypes.cast(arr, ctypes.POINTER(LayerCfg)))
    cfg._keep = arr  # keep the layer array alive with the struct
    return cfg


# ---------------------------------------------------------------- C names

def kvq_cache_bytes(cfg: Config) -> int:
    return int(load().kvq_cache_bytes(ctypes.byref(cfg)))


def kvq_create(cfg: Config, dev_buf: int, nbytes: int) -> int:
    h = ctypes.c_void_p()
    _check(load().kvq_create(ctypes.byref(cfg), ctypes.c_void_p(dev_buf), nbytes, ctypes.byref(h)), "kvq_create")
    return h.value


def kvq_append(h: int, layer: int, K: int, V: int, n_tokens: int, stream: int) -> None:
    _check(load().kvq_append(h, layer, K, V, n_tokens, stream), "kvq_append")


def kvq_decode_attn(h: int, layer: int, q: int, out: int, stream: int) -> None:
    _check(load().kvq_decode_attn(h, layer, q, out, stream), "kvq_decode_attn")


def kvq_decode_attn_noalloc(h: int, layer: int, q: int, out: int, stream: int) -> None:
    """kvq_decode_attn with the library's static device scratch: for callers
    that may not allocate device memory (see include/kvq.h)."""
    _check(load().kvq_decode_attn_noalloc(h, layer, q, out, stream), "kvq_decode_attn_noalloc")


def kvq_chunk_attn(h: int, layer: int, q: int, n_queries: int, out: int, workspace: int, workspace_bytes: int,
                   stream: int) -> None:
    _check(load().kvq_chunk_attn(h, layer, q, n_queries, out, workspace, workspace_bytes, stream), "kvq_chunk_attn")


def kvq_chunk_workspace_bytes(h: int) -> int:
    return int(load().kvq_chunk_workspace_bytes(h))


def kvq_decode_step(h: int, K: Sequence[int], V: Sequence[int], q: Sequence[int], out: Sequence[int],
                    stream: int) -> None:
    n = len(K)
    arr = [(ctypes.c_void_p * n)(*x) for x in (K, V, q, out)]
    _check(load().kvq_decode_step(h, *arr, stream), "kvq_decode_step")


def kvq_layer_view_get(h: int, layer: int) -> dict:
    v = LayerView()
    _check(load().kvq_layer_view_get(h, layer, ctypes.byref(v)), "kvq_layer_view_get")
    return {name: getattr(v, name) for name, _ in LayerView._fields_}


def kvq_equivalent_bits(h: int) -> float:
    return float(load().kvq_equivalent_bits(h))


def kvq_decode_bytes(h: int, layer: int) -> int:
    return int(load().kvq_decode_bytes(h, layer))


def kvq_device_error(h: int, stream: int) -> int:
    code = ctypes.c_int32(0)
    _check(load().kvq_device_error(h, ctypes.byref(code), stream), "kvq_device_error")
    return code.value


def kvq_selftest_bounded_wait(h: int, stream: int) -> None:
    _check(load().kvq_selftest_bounded_wait(h, stream), "kvq_selftest_bounded_wait")


def kvq_state_bytes(h: int) -> int:
    return int(load().kvq_state_bytes(h))


def kvq_state_save(h: int, dst: int, stream: int) -> None:
    _check(load().kvq_state_save(h, dst, stream), "kvq_state_save")


def kvq_state_restore(h: int, src: int, stream: int) -> None:
    _check(load().kvq_state_restore(h, src, stream), "kvq_state_restore")


def kvq_destroy(h: int) -> None:
    _check(load().kvq_destroy(h), "kvq_destroy")


def kvq_status_string(s: int) -> str:
    return load().kvq_status_string(s).decode()


# ---------------------------------------------------------------- convenience

def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dev_ptr(t, name: str, dtype, shape) -> int:
    import torch
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return int(t.data_ptr())


class KVQCache:
    """A layer-wise mixed-precision KV cache living in one torch-allocated
    device buffer."""

    def __init__(self, layers: Sequence[Tuple[int, int, int]], batch: int, num_q_heads: int,
                 num_kv_heads: int, head_dim: int, group_size: int, max_tokens: int, device="cuda"):
        import torch
        self.layers = [tuple(x) for x in layers]
        self.B, self.Hq, self.Hkv, self.D, self.G = batch, num_q_heads, num_kv_heads, head_dim, group_size
        self.max_tokens = max_tokens
        self.cfg = make_config(self.layers, batch, num_q_heads, num_kv_heads, head_dim, group_size, max_tokens)
        self.nbytes = kvq_cache_bytes(self.cfg)
        if self.nbytes == 0:
            raise KVQError(1, "kvq_cache_bytes")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.h = kvq_create(self.cfg, int(self.buf.data_ptr()), self.nbytes)

    def append(self, layer: int, K, V, stream=None) -> None:
        import torch
        n = K.shape[2]
        shp = (self.B, self.Hkv, n, self.D)
        kvq_append(self.h, layer, _dev_ptr(K, "K", torch.float16, shp), _dev_ptr(V, "V", torch.float16, shp),
                   n, _stream_ptr(stream))

    def decode_attn(self, layer: int, q, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((self.B, self.Hq, self.D), dtype=torch.float32, device=q.device)
        kvq_decode_attn(self.h, layer, _dev_ptr(q, "q", torch.float16, (self.B, self.Hq, self.D)),
                        _dev_ptr(out, "out", torch.float32, (self.B, self.Hq, self.D)), _stream_ptr(stream))
        return out

    def chunk_attn(self, layer: int, q, out=None, stream=None):
        """Causal attention of the queries of the newest q.shape[2] tokens:
        q fp16 [B, Hq, n, d] -> fp32 [B, Hq, n, d]."""
        import torch
        n = int(q.shape[2])
        shp = (self.B, self.Hq, n, self.D)
        if out is None:
            out = torch.empty(shp, dtype=torch.float32, device=q.device)
        if getattr(self, "_chunk_ws", None) is None:  # allocated on first use, kept with the cache
            self._chunk_ws = torch.empty(kvq_chunk_workspace_bytes(self.h), dtype=torch.uint8, device=self.buf.device)
        kvq_chunk_attn(self.h, layer, _dev_ptr(q, "q", torch.float16, shp), n,
                       _dev_ptr(out, "out", torch.float32, shp), int(self._chunk_ws.data_ptr()),
                       self._chunk_ws.numel(), _stream_ptr(stream))
        return out

    def decode_step(self, K: List, V: List, q: List, out: List, stream=None) -> None:
        import torch
        kv = (self.B, self.Hkv, 1, self.D)
        qs = (self.B, self.Hq, self.D)
        kvq_decode_step(self.h,
                        [_dev_ptr(x, "K", torch.float16, kv) for x in K],
                        [_dev_ptr(x, "V", torch.float16, kv) for x in V],
                        [_dev_ptr(x, "q", torch.float16, qs) for x in q],
                        [_dev_ptr(x, "out", torch.float32, qs) for x in out],
                        _stream_ptr(stream))

    def view(self, layer: int) -> dict:
        return kvq_layer_view_get(self.h, layer)

    def equivalent_bits(self) -> float:
        return kvq_equivalent_bits(self.h)

    def decode_bytes(self, layer: int) -> int:
        return kvq_decode_bytes(self.h, layer)

    def device_error(self, stream=None) -> int:
        return kvq_device_error(self.h, _stream_ptr(stream))

    def save_state(self, snapshot=None, stream=None):
        """Snapshot of the streaming state (token counters and FP16 windows of
        every layer) into a uint8 device tensor of kvq_state_bytes bytes,
        allocated if not given; returns it."""
        import torch
        n = kvq_state_bytes(self.h)
        if snapshot is None:
            snapshot = torch.empty(n, dtype=torch.uint8, device=self.buf.device)
        kvq_state_save(self.h, _dev_ptr(snapshot, "snapshot", torch.uint8, (n,)), _stream_ptr(stream))
        return snapshot

    def restore_state(self, snapshot, stream=None) -> None:
        import torch
        n = kvq_state_bytes(self.h)
        kvq_state_restore(self.h, _dev_ptr(snapshot, "snapshot", torch.uint8, (n,)), _stream_ptr(stream))

    def close(self) -> None:
        if getattr(self, "h", None):
            kvq_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
