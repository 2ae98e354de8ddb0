"""Intra-layer pruning of precision pairs by attention-output error.

KVTuner, section A2, "两阶段搜索空间剪枝算法" (two-stage search-space
pruning), step 1:
each layer's candidate KxVy pairs are scored by their equivalent bits and by
the relative attention-output error e_o = mean(|o - o_hat| / |o|) (defined
in its "A3 背景知识与关键观察" section, KV-cache quantization basics).  Pairs
not on the Pareto front of the two are dropped.  The page's example of what
survives in most layers is {KV8, K8V4, KV4, K4V2, KV2}.  This module does
not include the later stages: inter-layer clustering and the multi-objective
search, which is scored by model accuracy.

Everything here runs on the library's own kernels.  One cache is created with
one layer per candidate pair, plus a reference layer whose FP16 window is
longer than the calibration context.  None of the reference layer's tokens is
ever quantized, so its attention is the exact fp16-KV attention.  The
calibration K and V are appended to every layer, each query is decoded against
each layer, and e_o is reduced over the kernels' fp32 outputs.
"""

from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

from . import kvq

Pair = Tuple[int, int]
ALL_PAIRS: Tuple[Pair, ...] = tuple((kb, vb) for kb in (2, 3, 4, 8) for vb in (2, 3, 4, 8))
# the candidate set the pruning step starts from: {2, 4, 8} x {2, 4, 8}
KIVI_PAIRS: Tuple[Pair, ...] = tuple((kb, vb) for kb in (2, 4, 8) for vb in (2, 4, 8))


def pair_output_errors(K, V, queries: Sequence, pairs: Sequence[Pair] = KIVI_PAIRS, group_size: int = 32,
                       residual: int = 0, key_mode: int = kvq.KEY_PER_CHANNEL) -> Dict[Pair, float]:
    """e_o of every pair on one layer's calibration KV.

    K, V: [B, Hkv, T, D] fp16 CUDA tensors (one layer, T tokens).
    queries: [B, Hq, D] fp16 CUDA tensors, each attended over all T tokens.
    residual: FP16 window of the candidate layers (default group_size).
    Returns {(k_bits, v_bits): e_o}.  Per-token keys have no 3-bit kernel, so
    with key_mode KEY_PER_TOKEN a pair with k_bits = 3 raises ValueError."""
    import torch
    if not queries:
        raise ValueError("at least one query is needed")
    B, Hkv, T, D = (int(x) for x in K.shape)
    Hq = int(queries[0].shape[1])
    if T < 1:
        raise ValueError("calibration KV holds no token")
    pairs = [tuple(p) for p in pairs]
    if key_mode == kvq.KEY_PER_TOKEN and any(kb == 3 for kb, _ in pairs):
        raise ValueError("per-token keys have no 3-bit kernel")
    R = residual or group_size
    R_exact = group_size * (T // group_size + 1)  # longer than T: nothing is quantized
    layers = [(kb, vb, R, key_mode) for kb, vb in pairs] + [(8, 8, R_exact, kvq.KEY_PER_CHANNEL)]
    cache = kvq.KVQCache(layers, B, Hq, Hkv, D, group_size, T, device=K.device)
    try:
        for l in range(len(layers)):
            cache.append(l, K, V)
        ref = len(pairs)
        o = torch.stack([cache.decode_attn(ref, q) for q in queries])
        nz = o != 0
        o_nz = o[nz]
        errors = {}
        for i, p in enumerate(pairs):
            o_hat = torch.stack([cache.decode_attn(i, q) for q in queries])
            errors[p] = float(((o_hat[nz] - o_nz).abs() / o_nz.abs()).double().mean())
        code = cache.device_error()
        if code != 0:
            raise RuntimeError(f"pair_output_errors: device error word {code}")
        return errors
    finally:
        cache.close()


def equivalent_bits(pair: Pair) -> float:
    """Average bits per cached element of a pair: (k_bits + v_bits) / 2."""
    return (pair[0] + pair[1]) / 2


def pareto_front(errors: Dict[Pair, float]) -> List[Pair]:
    """The pairs that no other pair dominates, cheapest first.

    A pair is dominated when another has equivalent bits and e_o both no
    larger and at least one of them smaller."""
    keep = []
    for p, e in errors.items():
        b = equivalent_bits(p)
        if not any(equivalent_bits(q) <= b and f <= e and (equivalent_bits(q) < b or f < e)
                   for q, f in errors.items() if q != p):
            keep.append(p)
    return sorted(keep, key=lambda p: (equivalent_bits(p), errors[p]))


def prune_layer_pairs(K, V, queries: Sequence, pairs: Sequence[Pair] = KIVI_PAIRS, group_size: int = 32,
                      residual: int = 0, key_mode: int = kvq.KEY_PER_CHANNEL):
    """(front, errors): the layer's non-dominated pairs and every pair's e_o."""
    errors = pair_output_errors(K, V, queries, pairs, group_size, residual, key_mode)
    return pareto_front(errors), errors
