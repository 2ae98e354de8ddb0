"""Seeded synthetic workloads: per-layer precision tables and fp16 K/V/q generators.

This module holds no arithmetic of the quantization method itself.  It only
describes the six model-shaped workloads and draws their random inputs, so that
the CUDA path, the oracle, the tests and the benchmark all see the same bytes.

Distributions (stand-ins for real-model KV, which needs weights and datasets):

* keys  ``K[t, h, c] ~ N(mu_c, sigma_c)`` with ``mu_c ~ N(0, 0.5)`` (0.5 is the
  standard deviation) and ``sigma_c = exp(N(0, 0.5))``, both drawn per
  (layer, kv head, channel); a seeded pick of outlier channels per (layer, kv
  head) is multiplied by 10 or 20 (KIVI's observation that keys carry
  fixed per-channel outliers, "LLM 量化精读笔记 08", section 5.1);
* values ``V[t, h, c] ~ N(m_t, 1)`` with the mean drifting linearly from 0 to 4
  over all prefill and decode tokens (values drift over time, same page,
  section 5.2);
* queries ``q ~ N(0, 1)``.

All draws are fp32 rounded to fp16 (round to nearest even).  Generation uses
``torch.Generator`` on the requested device; the CPU and CUDA generators give
different streams for the same seed, so a test draws its inputs once, on one
device, and hands the same tensors to both sides.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

# (k_bits, v_bits, residual window R_l[, key mode[, RPC ratio in percent]])
LayerSpec = Tuple[int, ...]


def spec_fields(spec: Sequence[int]) -> Tuple[int, int, int, int, int]:
    """(k_bits, v_bits, R_l, key_mode, rpc_percent) of a layer spec; the key
    mode defaults to per channel (0) and the RPC ratio to 0 (a static window)."""
    kb, vb, r = spec[:3]
    km = spec[3] if len(spec) > 3 else 0
    rpc = spec[4] if len(spec) > 4 else 0
    return int(kb), int(vb), int(r), int(km), int(rpc)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    context: int          # prefill length S
    group_size: int       # key group G
    decode_steps: int
    n_outliers: int       # outlier key channels per (layer, kv head)
    outlier_factor: float
    seed: int
    layers: Tuple[LayerSpec, ...]

    @property
    def total_tokens(self) -> int:
        return self.context + self.decode_steps

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "layers": self.num_layers,
            "batch": self.batch,
            "q_heads": self.num_q_heads,
            "kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "context": self.context,
            "group_size": self.group_size,
            "decode_steps": self.decode_steps,
        }


def _uniform_pairs(n_layers: int, hi: Sequence[int], hi_pair, lo_pair, residual) -> Tuple[LayerSpec, ...]:
    out = []
    for l in range(n_layers):
        kb, vb = hi_pair if l in hi else lo_pair
        out.append((kb, vb, residual))
    return tuple(out)


def qwen_like_table(seed: int, n_layers: int = 28, residual: int = 64) -> Tuple[LayerSpec, ...]:
    """Seeded per-layer pairs from {K8V8, K8V4, K4V4, K4V2} whose mean equivalent
    bit width is exactly 4.0, with K8V8 forced on the first and last layer.

    Layers 1..n-2 start at K4V2 (3 bits); while their total is below the target,
    a uniformly drawn layer is raised one step along K4V2 -> K4V4 -> K8V4 -> K8V8
    (+1, +2, +2 bits), skipping a step that would overshoot.
    """
    ladder = [(4, 2), (4, 4), (8, 4), (8, 8)]
    eq = [3, 4, 6, 8]
    rng = np.random.Generator(np.random.PCG64(seed))
    level = [0] * n_layers
    inner = list(range(1, n_layers - 1))
    target_inner = 4 * n_layers - 2 * 8
    total = 3 * len(inner)
    guard = 0
    while total < target_inner:
        guard += 1
        if guard > 100000:
            raise RuntimeError("layer table search did not converge")
        l = inner[int(rng.integers(0, len(inner)))]
        if level[l] == len(ladder) - 1:
            continue
        step = eq[level[l] + 1] - eq[level[l]]
        if total + step > target_inner:
            continue
        level[l] += 1
        total += step
    out = []
    for l in range(n_layers):
        kb, vb = (8, 8) if l in (0, n_layers - 1) else ladder[level[l]]
        out.append((kb, vb, residual))
    return tuple(out)


def kvmix_table(seed: int, n_layers: int = 32, n_high: int = 6, context: int = 4096,
                group_size: int = 32, high_pair: Tuple[int, int] = (4, 3),
                ratios: Tuple[int, int] = (20, 10), dynamic: bool = True) -> Tuple[LayerSpec, ...]:
    """KVmix-style table: a seeded pick of high-precision layers (high_pair,
    K4V3 by default) and the rest K2V2.  Each layer's FP16 window starts at its
    RPC ratio (percent: 20 high, 10 low) of the prefill context, rounded down to
    whole key groups; with ``dynamic`` the ratio rides along as the fifth field
    and the window shrinks during decoding, otherwise it stays fixed."""
    rng = np.random.Generator(np.random.PCG64(seed))
    hi = set(int(x) for x in rng.choice(n_layers, n_high, replace=False))
    r_hi = group_size * ((ratios[0] * context) // (100 * group_size))
    r_lo = group_size * ((ratios[1] * context) // (100 * group_size))
    p_hi, p_lo = ratios if dynamic else (0, 0)
    return tuple((*high_pair, r_hi, 0, p_hi) if l in hi else (2, 2, r_lo, 0, p_lo) for l in range(n_layers))


def _make_workloads() -> List[Workload]:
    w1 = Workload("tiny-gqa-d64-K4V2", 1, 1, 8, 2, 64, 256, 32, 16, 2, 10.0, 1001,
                  ((4, 2, 32),))
    w2 = Workload("llama3.1-8b-shaped-decode", 32, 16, 32, 8, 128, 4096, 32, 128, 4, 10.0, 1002,
                  _uniform_pairs(32, {0, 1, 29, 30, 31}, (8, 4), (4, 2), 32))
    w3 = Workload("qwen2.5-7b-shaped-sensitive", 28, 32, 28, 4, 128, 8192, 64, 64, 8, 20.0, 1003,
                  qwen_like_table(1003))
    w4 = Workload("llama2-7b-shaped-kvmix-mha", 32, 30, 32, 32, 128, 4096, 32, 256, 4, 10.0, 1004,
                  kvmix_table(1004))
    w5 = Workload("llama2-70b-shaped-32k", 80, 8, 64, 8, 128, 32768, 128, 64, 4, 10.0, 1005,
                  _uniform_pairs(80, {0, 1, 77, 78, 79}, (8, 4), (4, 2), 128))
    # the KVmix page's own orientation: its averages (keys 2.19, values 2.38
    # bits) mean K3V4 on the high-precision layers, the mirror of w4's K4V3
    w6 = Workload("llama2-7b-shaped-kvmix-mha-k3v4", 32, 30, 32, 32, 128, 4096, 32, 256, 4, 10.0, 1006,
                  kvmix_table(1006, high_pair=(3, 4)))
    return [w1, w2, w3, w4, w5, w6]


WORKLOADS: List[Workload] = _make_workloads()


def workload(index: int) -> Workload:
    """Workloads are numbered 1..6 in the order they are listed above."""
    return WORKLOADS[index - 1]


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    return dataclasses.replace(w, **changes)


# --------------------------------------------------------------------------
# Random draws
# --------------------------------------------------------------------------

_PURPOSE = {"stats": 1, "k": 2, "v": 3, "q": 4}


def _gen(seed: int, layer: int, purpose: str, pos: int, device) -> torch.Generator:
    mixed = (seed * 1_000_003 + layer * 10_007 + _PURPOSE[purpose] * 101 + pos * 7) % (2**62)
    g = torch.Generator(device=device)
    g.manual_seed(mixed)
    return g


@dataclasses.dataclass
class KeyStats:
    mu: torch.Tensor      # [Hkv, d] fp32
    sigma: torch.Tensor   # [Hkv, d] fp32
    scale: torch.Tensor   # [Hkv, d] fp32, 1 or the outlier factor


def key_stats(w: Workload, layer: int, device="cpu") -> KeyStats:
    g = _gen(w.seed, layer, "stats", 0, device)
    shape = (w.num_kv_heads, w.head_dim)
    mu = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 0.5
    sigma = torch.exp(torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 0.5)
    scale = torch.ones(shape, device=device, dtype=torch.float32)
    if w.n_outliers > 0:
        keys = torch.rand(shape, generator=g, device=device)
        idx = torch.argsort(keys, dim=1)[:, : w.n_outliers]
        scale.scatter_(1, idx, w.outlier_factor)
    return KeyStats(mu, sigma, scale)


def gen_kv(w: Workload, layer: int, start: int, n: int, device="cpu",
           stats: Optional[KeyStats] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """K and V for token positions [start, start+n) of one layer, fp16,
    shape [B, Hkv, n, d], contiguous."""
    if stats is None:
        stats = key_stats(w, layer, device)
    B, H, d = w.batch, w.num_kv_heads, w.head_dim
    gk = _gen(w.seed, layer, "k", start, device)
    z = torch.randn((B, H, n, d), generator=gk, device=device, dtype=torch.float32)
    k = (stats.mu[None, :, None, :] + stats.sigma[None, :, None, :] * z) * stats.scale[None, :, None, :]
    gv = _gen(w.seed, layer, "v", start, device)
    t = torch.arange(start, start + n, device=device, dtype=torch.float32)
    denom = max(w.total_tokens - 1, 1)
    m = 4.0 * t / denom
    v = torch.randn((B, H, n, d), generator=gv, device=device, dtype=torch.float32) + m[None, None, :, None]
    return k.to(torch.float16).contiguous(), v.to(torch.float16).contiguous()


def gen_q(w: Workload, layer: int, step: int, device="cpu") -> torch.Tensor:
    """Query for one decode step of one layer, fp16, shape [B, Hq, d]."""
    g = _gen(w.seed, layer, "q", step, device)
    q = torch.randn((w.batch, w.num_q_heads, w.head_dim), generator=g, device=device,
                    dtype=torch.float32)
    return q.to(torch.float16).contiguous()
