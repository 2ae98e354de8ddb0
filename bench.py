"""Benchmark: mixed-precision KV decode attention on one GB300 (or N replicas).

A step is one decode step of the whole hot path over every layer of the
workload: append the new token (FP16 window; a group flush with quantize +
pack every G steps) and run decode attention over the quantized cache plus
the window.  The default workload is the Llama-3.1-8B-shaped decode: 32
layers, 32 q / 8 kv heads, head_dim 128, batch 16, context 4096, G = R = 32,
K8V4 on layers 0-1 and 29-31 and K4V2 elsewhere.

Reported:
  value       decode tokens/s (batch x ranks / step time), device-timed with
              CUDA events around K replays of the step's CUDA graph
  e2e         the same metric through KVQCache.decode_step with every step's
              inputs copied from pinned host memory and its outputs read back
  roofline    decode-attention kernel: algorithmic bytes per launch / average
              launch duration (a second timed pass replaying a decode-only
              graph of all layers) against the measured HBM copy bandwidth
  cpu_baseline  the oracle timed on the host cores on a bounded sample

--impl reference times the oracle (the plain CPU statement of the method) on
the same workload, one bounded sample per step.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "mixed-precision KV decode-attn tokens/s; cache-read GB/s as % of HBM peak"
L2_BYTES = 129 * 1024 * 1024  # GB300 L2: a step reading more than this cannot be served from it


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while it runs."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.samples = []
        self.windows = []
        self._proc = None
        self._thr = None
        self.gpu_index = gpu_index
        self.interval_ms = interval_ms

    def start(self):
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self._proc = None
            return
        self._thr = threading.Thread(target=self._read, daemon=True)
        self._thr.start()

    def _read(self):
        for line in self._proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self._proc is None:
            return None
        self._proc.terminate()
        try:
            self._proc.wait(timeout=5)
        except Exception:
            self._proc.kill()
        if self._thr:
            self._thr.join(timeout=2)
        inside = [s for t, s in self.samples if any(a - 0.05 <= t <= b + 0.05 for a, b in self.windows)]
        use = inside or [s for _, s in self.samples]
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in use:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "in_timed_region": bool(inside)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (timings: the slowest rank sets the
    job's time).  NCCL reduces on the rank's GPU, gloo on the host."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------
# CPU oracle timing (bounded sample)
# ----------------------------------------------------------------------------

class OracleSampler:
    """Times the oracle's decode step (append one token, then fp64 attention
    over the dequantized cache) for one (batch, kv head) unit of each distinct
    precision pair, at full context, and extrapolates to the whole step
    (all units of all layers).  The oracle runs as it stands, single-threaded
    numpy."""

    def __init__(self, w):
        from mixed_precision_quantized_quant_gb300 import workloads as W
        from oracle import kvq_oracle as O
        self.W, self.w = W, w
        seen, self.layers = set(), []
        for l, p in enumerate(w.layers):
            if p not in seen:
                seen.add(p)
                self.layers.append(l)
        self.unit_w = W.scaled(w, batch=1, num_kv_heads=1, num_q_heads=w.num_q_heads // w.num_kv_heads)
        self.caches = {}
        for l in self.layers:
            kb, vb, R = w.layers[l][:3]
            km = w.layers[l][3] if len(w.layers[l]) > 3 else 0
            ora = O.OracleLayerCache(1, 1, w.head_dim, w.group_size, kb, vb, R, km)
            k, v = W.gen_kv(self.unit_w, l, 0, w.context)
            ora.append(k.numpy(), v.numpy())
            self.caches[l] = ora
        self.pos = 0
        U = w.batch * w.num_kv_heads
        self.count = {l: sum(1 for p in w.layers if p == w.layers[l]) * U for l in self.layers}
        self.desc = (f"oracle decode step (append 1 token + fp64 attention over the dequantized cache) "
                     f"for 1 of {U} (batch, kv head) units on layers {self.layers} (one per distinct "
                     f"precision pair) at context {w.context}; per-unit time x {U} units x "
                     f"{w.num_layers} layers")

    def errors(self):
        """Quantization error of each distinct precision pair on the sampled
        unit (KVTuner A3's metrics): e_k, e_v over the quantized tokens,
        e_a = mean |a - a_hat| of the attention weights and e_o of the output
        for the first query, against fp64 over the fp16 K and V."""
        import numpy as np
        from oracle import kvq_oracle as O
        out = {}
        for l in self.layers:
            kb, vb = self.w.layers[l][:2]
            ora = self.caches[l]
            kh, vh = ora.dequantized(0)
            k, v = (x.numpy()[0, 0].astype(np.float64) for x in self.W.gen_kv(self.unit_w, l, 0, self.w.context))
            nq = ora.n_q
            q = self.W.gen_q(self.unit_w, l, 0).numpy()[0].astype(np.float64)
            T = kh.shape[0]
            ea, o_ref, o_hat = [], [], []
            for h in range(q.shape[0]):
                def weights(kk):
                    x = kk[:T] @ q[h] / np.sqrt(kk.shape[1])
                    e = np.exp(x - x.max())
                    return e / e.sum()
                a, ah = weights(k), weights(kh)
                ea.append(np.abs(a - ah).mean())
                o_ref.append(O.attention_fp64(q[h], k[:T], v[:T]))
                o_hat.append(O.attention_fp64(q[h], kh, vh))
            out[f"K{kb}V{vb}"] = {"e_k": round(O.rel_error(k[:nq], kh[:nq]), 5),
                                  "e_v": round(O.rel_error(v[:nq], vh[:nq]), 5),
                                  "e_a": float(f"{np.mean(ea):.3e}"),
                                  "e_o": round(O.rel_error(np.stack(o_ref), np.stack(o_hat)), 5)}
        return out

    def step(self) -> float:
        """Seconds one full decode step would take, from one timed unit-step
        per distinct layer type."""
        total = 0.0
        for l in self.layers:
            k1, v1 = self.W.gen_kv(self.unit_w, l, self.w.context + self.pos, 1)
            q = self.W.gen_q(self.unit_w, l, self.pos).numpy()
            t0 = time.perf_counter()
            self.caches[l].append(k1.numpy(), v1.numpy())
            self.caches[l].attend(q)
            total += (time.perf_counter() - t0) * self.count[l]
        self.pos += 1
        return total


def oracle_sample(w, budget_s: float = 12.0):
    """(tokens/s, seconds per full step, description, quantization errors)
    from repeated sampled steps until about budget_s seconds of oracle work."""
    smp = OracleSampler(w)
    errors = smp.errors()
    t_start = time.perf_counter()
    steps = []
    while len(steps) < 3 or (time.perf_counter() - t_start < budget_s and len(steps) < 64):
        steps.append(smp.step())
    step_s = statistics.median(steps)
    return w.batch / step_s, step_s, smp.desc + f"; median over {len(steps)} sampled steps", errors


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def _with_key_mode(w, args):
    """The workload with every layer's keys in the requested mode (per token:
    KVTuner's per-token-asym mode; 2, 4 or 8-bit keys only)."""
    if args.key_mode == "channel":
        return w
    from mixed_precision_quantized_quant_gb300 import workloads as W
    if any(l[0] == 3 for l in w.layers):
        raise SystemExit("per-token keys need 2, 4 or 8-bit keys; this workload has 3-bit keys")
    return W.scaled(w, name=w.name + "-per-token-keys", layers=tuple((kb, vb, r, 1) for kb, vb, r in w.layers))


def run_gpu(args):
    import numpy as np
    import torch

    from mixed_precision_quantized_quant_gb300 import kvq as K
    from mixed_precision_quantized_quant_gb300 import workloads as W

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K.load()
    w = _with_key_mode(W.workload(args.workload), args)
    if args.layers:  # profiling runs: the workload's first N layers
        w = W.scaled(w, num_layers=args.layers, layers=tuple(w.layers[:args.layers]))
    L, B, Hq, Hkv, D = w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    steps, warm = args.steps, args.warmup
    cap = w.context + warm + steps
    stream = torch.cuda.Stream(device=dev)

    cache = K.KVQCache(w.layers, B, Hq, Hkv, D, w.group_size, cap, device=dev)

    # ---- prefill (timed separately: append GB/s)
    prefill_ms = 0.0
    prefill_bytes = 0
    with torch.cuda.stream(stream):
        for l in range(L):
            k, v = W.gen_kv(w, l, 0, w.context, device=dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            cache.append(l, k, v, stream=stream)
            e1.record(stream)
            stream.synchronize()
            prefill_ms += e0.elapsed_time(e1)
            vw = cache.view(l)
            U = B * Hkv
            prefill_bytes += (k.numel() + v.numel()) * 2 + U * (vw["quantized_tokens"] // w.group_size) * \
                vw["record_bytes"] + U * vw["residual_tokens"] * 4 * D
            del k, v

    # ---- per-step inputs, resident in HBM
    nst = warm + steps
    kin = torch.empty((nst, L, B, Hkv, 1, D), dtype=torch.float16, device=dev)
    vin = torch.empty_like(kin)
    qin = torch.empty((nst, L, B, Hq, D), dtype=torch.float16, device=dev)
    for s in range(nst):
        for l in range(L):
            k1, v1 = W.gen_kv(w, l, w.context + s, 1, device=dev)
            kin[s, l].copy_(k1)
            vin[s, l].copy_(v1)
            qin[s, l].copy_(W.gen_q(w, l, s, device=dev))
    outs = torch.empty((L, B, Hq, D), dtype=torch.float32, device=dev)
    # inputs are staged into fixed buffers so the step graph is captured once
    k_cur = torch.empty((L, B, Hkv, 1, D), dtype=torch.float16, device=dev)
    v_cur = torch.empty_like(k_cur)
    q_cur = torch.empty((L, B, Hq, D), dtype=torch.float16, device=dev)
    torch.cuda.synchronize()

    def step_lists():
        return ([k_cur[l] for l in range(L)], [v_cur[l] for l in range(L)], [q_cur[l] for l in range(L)],
                [outs[l] for l in range(L)])

    Ks, Vs, Qs, Os = step_lists()

    def run_step(s):
        k_cur.copy_(kin[s], non_blocking=True)
        v_cur.copy_(vin[s], non_blocking=True)
        q_cur.copy_(qin[s], non_blocking=True)
        cache.decode_step(Ks, Vs, Qs, Os, stream=stream)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for s in range(warm):
            run_step(s)
        stream.synchronize()
        _barrier(world)
        torch.cuda.synchronize()
        bytes_step = sum(cache.decode_bytes(l) for l in range(L))  # at the first timed step
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        ev0.record(stream)
        for s in range(warm, warm + steps):
            run_step(s)
        ev1.record(stream)
        stream.synchronize()
        t1 = time.time()
        sampler.mark(t0, t1)
        torch.cuda.synchronize()
        _barrier(world)
    ms_total = ev0.elapsed_time(ev1)
    ms_total = _max_over_ranks(ms_total, world)
    ms_step = ms_total / steps
    tokens_per_s = world * B * steps / (ms_total / 1e3)
    gpu_launches = steps * 2 * L

    # ---- decode-attention roofline: replay a decode-only graph of all layers
    dec_bytes = [cache.decode_bytes(l) for l in range(L)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for l in range(L):  # warm (and loads every instantiation before capture)
            cache.decode_attn(l, q_cur[l], outs[l], stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                cache.decode_attn(l, q_cur[l], outs[l], stream=torch.cuda.current_stream())
        for _ in range(3):
            g.replay()
        stream.synchronize()
        reps = max(10, min(200, int(200 / max(ms_step, 0.05))))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
        sampler.mark(t0, time.time())
    dec_ms_per_launch = e0.elapsed_time(e1) / reps / L
    dec_bytes_per_launch = sum(dec_bytes) / L
    clocks = sampler.stop()

    # ---- end to end through the public API, pinned host copies every step
    e2e_tps = None
    e2e_cache = None
    if not args.no_e2e:
        h_k = torch.empty((nst, L, B, Hkv, 1, D), dtype=torch.float16).pin_memory()
        h_v = torch.empty_like(h_k).pin_memory()
        h_q = torch.empty((nst, L, B, Hq, D), dtype=torch.float16).pin_memory()
        h_k.copy_(kin.cpu())
        h_v.copy_(vin.cpu())
        h_q.copy_(qin.cpu())
        h_out = torch.empty((2, L, B, Hq, D), dtype=torch.float32).pin_memory()  # two readback slots
        e2e_cache = K.KVQCache(w.layers, B, Hq, Hkv, D, w.group_size, cap, device=dev)
        with torch.cuda.stream(stream):
            for l in range(L):
                k, v = W.gen_kv(w, l, 0, w.context, device=dev)
                e2e_cache.append(l, k, v, stream=stream)
                del k, v
            stream.synchronize()
        # Pipelined through the public API: step s+1's inputs are uploaded
        # from pinned memory on a copy stream while step s computes, and step
        # s's outputs are staged on the device and read back while step s+1
        # runs.  Every step still copies its inputs in and its outputs out.
        copy = torch.cuda.Stream(device=dev)
        st_k = [torch.empty_like(k_cur) for _ in range(2)]
        st_v = [torch.empty_like(v_cur) for _ in range(2)]
        st_q = [torch.empty_like(q_cur) for _ in range(2)]
        st_o = [torch.empty_like(outs) for _ in range(2)]
        up = [torch.cuda.Event() for _ in range(2)]     # inputs of a slot uploaded
        used = [torch.cuda.Event() for _ in range(2)]   # inputs of a slot consumed by the step
        done = [torch.cuda.Event() for _ in range(2)]   # outputs of a slot staged
        down = [torch.cuda.Event() for _ in range(2)]   # outputs of a slot read back

        def upload(s):
            b = s & 1
            with torch.cuda.stream(copy):
                copy.wait_event(used[b])
                st_k[b].copy_(h_k[s], non_blocking=True)
                st_v[b].copy_(h_v[s], non_blocking=True)
                st_q[b].copy_(h_q[s], non_blocking=True)
                up[b].record(copy)

        def run(s, n):
            upload(s)
            for i in range(s, s + n):
                b = i & 1
                if i + 1 < s + n:
                    upload(i + 1)
                with torch.cuda.stream(stream):
                    stream.wait_event(up[b])
                    k_cur.copy_(st_k[b], non_blocking=True)
                    v_cur.copy_(st_v[b], non_blocking=True)
                    q_cur.copy_(st_q[b], non_blocking=True)
                    used[b].record(stream)
                    e2e_cache.decode_step(Ks, Vs, Qs, Os, stream=stream)
                    stream.wait_event(down[b])  # the slot's previous readback has finished
                    st_o[b].copy_(outs, non_blocking=True)
                    done[b].record(stream)
                with torch.cuda.stream(copy):
                    copy.wait_event(done[b])
                    h_out[b].copy_(st_o[b], non_blocking=True)  # slot b's previous result was synced
                    down[b].record(copy)
                if i >= s + 1:
                    down[(i - 1) & 1].synchronize()  # step i-1's result is on the host
            down[(s + n - 1) & 1].synchronize()

        run(0, warm)
        _barrier(world)
        t0 = time.perf_counter()
        run(warm, steps)
        t1 = time.perf_counter()
        _barrier(world)
        e2e_s = _max_over_ranks(t1 - t0, world)
        e2e_tps = world * B * steps / e2e_s
    h2d = L * (2 * B * Hkv * D * 2 + B * Hq * D * 2)
    d2h = L * B * Hq * D * 4
    err = cache.device_error(stream) | (e2e_cache.device_error(stream) if e2e_cache is not None else 0)
    if err:
        raise RuntimeError(f"device error word {err}")

    peak, peak_kind = _peaks()
    achieved = dec_bytes_per_launch / (dec_ms_per_launch / 1e3) / 1e9
    # the committed capture covers every layer of the workload: no figure for a layer subset
    traffic = None if args.layers else _ncu_traffic(w.name)
    result = {
        "metric": METRIC,
        "value": round(tokens_per_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 codes/fp32 accumulate",
        "data": "synthetic (seeded: keys N(mu_c, sigma_c) with channel outliers, values with drifting mean)",
        "config": {**w.describe(), "equivalent_bits": round(cache.equivalent_bits(), 5),
                   "parallelism": f"replicas x{world} (independent (batch, kv head) units, no collective)",
                   "l2": ("inputs larger than L2: %.2f GB of cache read per step" % (bytes_step / 1e9)
                          if bytes_step > L2_BYTES else
                          "cache smaller than L2 (%.3f MB read per step), not flushed: a latency figure"
                          % (bytes_step / 1e6))},
        "cache_read_gbs": round(bytes_step / (ms_step / 1e3) / 1e9, 1),
        "cache_read_frac_of_peak": round(bytes_step / (ms_step / 1e3) / 1e9 / peak, 4),
        "append_prefill_gbs": round(prefill_bytes / (prefill_ms / 1e3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "decode_kernel (all layers, decode-only graph replay)",
                     "bytes_per_launch": int(dec_bytes_per_launch),
                     "us_per_launch": round(dec_ms_per_launch * 1e3, 3),
                     "peak_source": f"{peak_kind} HBM copy bandwidth"},
        "e2e": None if e2e_tps is None else {"value": round(e2e_tps, 1), "unit": "tokens/s",
                                             "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        tps, step_s, desc, errors = oracle_sample(w, budget_s=args.cpu_budget)
        result["cpu_baseline"] = {"value": round(tps, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                  "sample": desc, "seconds_per_step": round(step_s, 2)}
        result["quant_error"] = {"per_pair": errors,
                                 "of": "one sampled (batch, kv head) unit at full context, first query; "
                                       "e_k, e_v over its quantized tokens, e_a and e_o against fp64 "
                                       "attention over the fp16 K and V (KVTuner A3)"}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def _ncu_traffic(workload_name):
    """Mean DRAM bytes (read + write) per decode launch of one step, from the
    committed ncu summary of this workload, if it was taken on the current
    decode kernel source (its sha256 prefix is recorded in the summary)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"decode_kernel_dram_{workload_name}.txt")
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith((" ", "#", "|")):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        src = os.path.join(ROOT, "mixed_precision_quantized_quant_gb300", "csrc", "kvq_decode.cuh")
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if kv.get("kernel_source_sha256_16") != h:
            return None
        return int(float(kv["dram_bytes_per_launch_mean"]))
    except (OSError, KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
# chunk attention (causal prefill over the quantized cache)
# ----------------------------------------------------------------------------

CHUNK_METRIC = "causal chunk attention over the quantized cache, TFLOP/s (4 d per visible (query, key) pair)"


def _chunk_flops(B, Hq, D, T, n):
    """Algorithmic FLOPs of one layer: 2 d for q.k and 2 d for p.v per visible pair."""
    visible = n * (T - n) + n * (n + 1) // 2
    return 4.0 * D * visible * Hq * B


def _chunk_workload(args):
    from mixed_precision_quantized_quant_gb300 import workloads as W
    w = _with_key_mode(W.workload(args.workload), args)
    w = W.scaled(w, batch=args.chunk_batch)
    if args.layers:
        w = W.scaled(w, num_layers=args.layers, layers=tuple(w.layers[:args.layers]))
    n = args.chunk or w.context
    return w, n


class ChunkOracleSampler:
    """Times the oracle's chunk attention (fp64 over the dequantized cache) for
    the last `rows` queries of the chunk on one (batch, kv head) unit of each
    distinct precision pair, and scales by visible pairs to the whole step."""

    def __init__(self, w, n, rows=8):
        import numpy as np
        from mixed_precision_quantized_quant_gb300 import workloads as W
        from oracle import kvq_oracle as O
        self.w, self.n, self.rows = w, n, rows
        T, D, rep = w.context, w.head_dim, w.num_q_heads // w.num_kv_heads
        seen, self.layers = set(), []
        for l, p in enumerate(w.layers):
            if p not in seen:
                seen.add(p)
                self.layers.append(l)
        uw = W.scaled(w, batch=1, num_kv_heads=1, num_q_heads=rep)
        self.caches, self.q = {}, {}
        rng = np.random.default_rng(7)
        for l in self.layers:
            kb, vb, R = w.layers[l][:3]
            km = w.layers[l][3] if len(w.layers[l]) > 3 else 0
            ora = O.OracleLayerCache(1, 1, D, w.group_size, kb, vb, R, km)
            k, v = W.gen_kv(uw, l, 0, T)
            ora.append(k.numpy(), v.numpy())
            self.caches[l] = ora
            self.q[l] = rng.standard_normal((1, rep, rows, D)).astype(np.float16)
        self.count = {l: sum(1 for p in w.layers if p == w.layers[l]) for l in self.layers}
        # the sample's queries are the last `rows` positions: each sees about T keys
        self.sample_flops = {l: 4.0 * D * rep * sum(T - rows + i + 1 for i in range(rows)) for l in self.layers}
        self.step_flops = w.num_layers * _chunk_flops(w.batch, w.num_q_heads, D, T, n)
        self.desc = (f"oracle chunk attention (fp64 over the dequantized cache) for the last {rows} queries x "
                     f"{rep} heads of 1 (batch, kv head) unit on layers {self.layers} (one per distinct "
                     f"precision pair) at context {T}; time per visible pair scaled to the step's "
                     f"{self.step_flops / 4 / D:.3g} pairs")

    def step(self) -> float:
        """Seconds one full chunk step would take (all layers, all units)."""
        secs, flops = 0.0, 0.0
        for l in self.layers:
            c = self.caches[l]
            t0 = time.perf_counter()
            c.attend_chunk(self.q[l])  # the queries of the newest `rows` tokens
            secs += (time.perf_counter() - t0) * self.count[l]
            flops += self.sample_flops[l] * self.count[l]
        return secs * self.step_flops / flops


def chunk_oracle_sample(w, n, budget_s):
    smp = ChunkOracleSampler(w, n)
    t_start = time.perf_counter()
    steps = []
    while len(steps) < 2 or (time.perf_counter() - t_start < budget_s and len(steps) < 16):
        steps.append(smp.step())
    step_s = statistics.median(steps)
    return smp.step_flops / step_s / 1e12, step_s, smp.desc + f"; median over {len(steps)} samples"


def _tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_chunk(args):
    import torch

    from mixed_precision_quantized_quant_gb300 import kvq as K
    from mixed_precision_quantized_quant_gb300 import workloads as W

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K.load()
    w, n = _chunk_workload(args)
    L, B, Hq, Hkv, D, T = w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.context
    stream = torch.cuda.Stream(device=dev)
    cache = K.KVQCache(w.layers, B, Hq, Hkv, D, w.group_size, T, device=dev)
    with torch.cuda.stream(stream):
        for l in range(L):
            k, v = W.gen_kv(w, l, 0, T, device=dev)
            cache.append(l, k, v, stream=stream)
            del k, v
        stream.synchronize()
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    q = torch.randn((B, Hq, n, D), generator=gen, device=dev).half()
    out = torch.empty((B, Hq, n, D), dtype=torch.float32, device=dev)
    flops_layer = _chunk_flops(B, Hq, D, T, n)

    def run_step():
        for l in range(L):
            cache.chunk_attn(l, q, out, stream=stream)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run_step()
        stream.synchronize()
        _barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        ev0.record(stream)
        for _ in range(args.steps):
            run_step()
        ev1.record(stream)
        stream.synchronize()
        sampler.mark(t0, time.time())
        torch.cuda.synchronize()
        _barrier(world)
    ms_total = _max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_step = ms_total / args.steps
    tflops = world * L * flops_layer * args.steps / (ms_total / 1e3) / 1e12
    clocks = sampler.stop()

    # end to end: each layer's queries copied from pinned host memory, outputs read back
    e2e = None
    if not args.no_e2e:
        h_q = q.cpu().pin_memory()
        h_out = torch.empty((2, B, Hq, n, D), dtype=torch.float32).pin_memory()  # two readback slots
        # Pipelined: layer l+1's queries are uploaded on a copy stream while
        # layer l computes, and layer l's outputs are read back while layer
        # l+1 computes (two device slots each); every layer still copies its
        # queries in and its outputs out.
        copy = torch.cuda.Stream(device=dev)
        q_dev = [torch.empty_like(q) for _ in range(2)]
        o_dev = [torch.empty_like(out) for _ in range(2)]
        up = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        down = [torch.cuda.Event() for _ in range(2)]

        def upload(i):
            b = i & 1
            with torch.cuda.stream(copy):
                copy.wait_event(used[b])
                q_dev[b].copy_(h_q, non_blocking=True)
                up[b].record(copy)

        def e2e_step():
            upload(0)
            for l in range(L):
                b = l & 1
                if l + 1 < L:
                    upload(l + 1)
                with torch.cuda.stream(stream):
                    stream.wait_event(up[b])
                    stream.wait_event(down[b])  # the slot's previous readback has finished
                    cache.chunk_attn(l, q_dev[b], o_dev[b], stream=stream)
                    used[b].record(stream)
                    done[b].record(stream)
                with torch.cuda.stream(copy):
                    copy.wait_event(done[b])
                    h_out[b].copy_(o_dev[b], non_blocking=True)
                    down[b].record(copy)
                if l >= 1:
                    down[(l - 1) & 1].synchronize()  # layer l-1's result is on the host
            down[(L - 1) & 1].synchronize()

        for _ in range(min(args.warmup, 3)):
            e2e_step()
        _barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        t1 = time.perf_counter()
        _barrier(world)
        e2e_s = _max_over_ranks(t1 - t0, world)
        e2e = {"value": round(world * L * flops_layer * args.steps / e2e_s / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": L * q.numel() * 2, "d2h_bytes_per_step": L * out.numel() * 4}
    if cache.device_error(stream):
        raise RuntimeError("device error word set")
    peak, kind = _tensor_peak()
    achieved = flops_layer / (ms_step / L / 1e3) / 1e12
    result = {
        "metric": CHUNK_METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 MMA operands (hi + lo halves)/fp32 accumulate",
        "data": "synthetic (seeded: keys N(mu_c, sigma_c) with channel outliers, values with drifting mean)",
        "config": {**w.describe(), "op": "chunk attention", "chunk_queries": n,
                   "equivalent_bits": round(cache.equivalent_bits(), 5),
                   "parallelism": f"replicas x{world}",
                   "l2": "compute-bound; the quantized cache of a layer is L2-resident and read by every CTA of its unit"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "chunk_attn_kernel (all layers)", "flops_per_launch": flops_layer,
                     "us_per_launch": round(ms_step / L * 1e3, 2),
                     "peak_source": f"{kind} bf16 dense (fp16 has the same tensor rate); the kernel issues two "
                                    f"MMAs (hi, lo) per algorithmic product"},
        "e2e": e2e, "gpu_launches": L * args.steps, "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        tf, step_s, desc = chunk_oracle_sample(w, n, args.cpu_budget)
        result["cpu_baseline"] = {"value": round(tf, 8), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                  "sample": desc, "seconds_per_step": round(step_s, 1)}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


# ----------------------------------------------------------------------------
# reference arm: the oracle
# ----------------------------------------------------------------------------

def run_reference(args):
    from mixed_precision_quantized_quant_gb300 import workloads as W
    world, rank, _ = _dist()
    if rank != 0:
        return
    w = _with_key_mode(W.workload(args.workload), args)
    smp = OracleSampler(w)
    vals = []
    for s in range(args.warmup + args.steps):
        step_s = smp.step()
        if s >= args.warmup:
            vals.append(step_s)
    step_s = statistics.median(vals)
    v = w.batch / step_s
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": round(v, 6), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 quantizer / f64 attention",
        "data": "synthetic", "config": w.describe(),
        "cpu_baseline": {"value": round(v, 6), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": smp.desc + "; each step is one sampled unit-step per layer type"},
        "e2e": {"value": round(v, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_chunk_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    w, n = _chunk_workload(args)
    smp = ChunkOracleSampler(w, n)
    vals = []
    for s in range(args.warmup + args.steps):
        step_s = smp.step()
        if s >= args.warmup:
            vals.append(step_s)
    step_s = statistics.median(vals)
    v = smp.step_flops / step_s / 1e12
    print(json.dumps({
        "impl": "reference", "metric": CHUNK_METRIC, "value": round(v, 8), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 quantizer / f64 attention", "data": "synthetic",
        "config": {**w.describe(), "op": "chunk attention", "chunk_queries": n},
        "cpu_baseline": {"value": round(v, 8), "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": smp.desc},
        "e2e": {"value": round(v, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=120)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", type=int, default=2, help="1..5; 2 is the Llama-3.1-8B-shaped decode")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="profiling runs: skip the end-to-end leg")
    ap.add_argument("--layers", type=int, default=0, help="profiling runs: only the workload's first N layers")
    ap.add_argument("--key-mode", choices=["channel", "token"], default="channel",
                    help="keys per channel over groups (KIVI) or per token (per-token-asym) on every layer")
    ap.add_argument("--op", choices=["decode", "chunk"], default="decode",
                    help="decode: the per-token decode step; chunk: causal chunk attention of n queries "
                         "over every layer's quantized cache (prefill over the dequantized cache)")
    ap.add_argument("--chunk", type=int, default=0, help="--op chunk: queries per chunk (default: the context)")
    ap.add_argument("--chunk-batch", type=int, default=2, help="--op chunk: sequences")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.op == "chunk" and args.steps == 120:
        args.steps = 5  # a chunk step is a whole-model prefill attention
    if args.impl == "reference":
        run_chunk_reference(args) if args.op == "chunk" else run_reference(args)
    elif args.op == "chunk":
        run_chunk(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
