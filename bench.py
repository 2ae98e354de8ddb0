"""Benchmark: mixed-precision KV decode attention on one GB300 (or N replicas).

A step is one decode step of the whole hot path over every layer of the
workload: append the new token (FP16 window; a group flush with quantize +
pack when a layer's window fills) and run decode attention over the quantized
cache plus the window.  The default workload is the largest one, the
Llama-2-70B-shaped 32K-context decode: 80 layers, 64 q / 8 kv heads, head_dim
128, batch 8, G = R = 128, K8V4 on layers 0-1 and 77-79 and K4V2 elsewhere.
The prefill stops short of the context by the offset that makes the middle
timed step flush a key group on every layer, so the quantize + pack half of
the decode step is inside the timed window whatever --steps is.

Reported:
  value       decode tokens/s (batch x ranks x steps / time), device-timed
              with CUDA events around the K timed replays of the step's CUDA
              graph (an event after each step gives the per-step times; the
              flush step is reported separately)
  e2e         the same metric through KVQCache.decode_step with every step's
              inputs copied from pinned host memory and its outputs read back
  roofline    decode-attention kernel: algorithmic bytes per launch / launch
              duration, from a second pass replaying a decode-only graph of
              all layers (median of >= 10 replays, one event pair each)
              against the measured HBM copy bandwidth
  other_workloads  the same figures (no end-to-end leg) for --extra-workloads
  cpu_baseline  the oracle on the host cores (one worker process per core) on
              a bounded sample of the step's (layer, unit) pairs

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
# CPU oracle timing (bounded sample, one worker process per host core)
# ----------------------------------------------------------------------------

def _oracle_worker(conn, jobs):
    """One host core: prefill the oracle caches of its (layer, unit) pairs,
    then run a decode step on each of them per request (append the step's
    token, then fp64 attention over the dequantized cache)."""
    from oracle import kvq_oracle as O
    caches = []
    for d, G, kb, vb, R, km, rpc, k, v in jobs:
        c = O.OracleLayerCache(1, 1, d, G, kb, vb, R, km, rpc)
        c.append(k, v)
        caches.append(c)
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg is None:
            break
        for c, (k1, v1, q) in zip(caches, msg):
            c.append(k1, v1)
            c.attend(q)
        conn.send("done")
    conn.close()


class OracleSampler:
    """Times the oracle's decode step on a bounded sample of the workload: n_s
    of the step's L x U (layer, (batch, kv head) unit) pairs, on layers spread
    evenly over the model (so the precision pairs appear in about their
    proportions), each at the full prefill length.  Each pair lives in one of
    `procs` worker processes (spawned, one host core each, single-threaded
    numpy); a sample step sends every worker its pairs' next token and query
    and waits for all of them.  The oracle runs as it stands.

    tokens/s = batch x (n_s / (L x U)) / (wall time of a sample step)."""

    def __init__(self, w, prefill=None, procs=None):
        import multiprocessing as mp
        import numpy as np
        from mixed_precision_quantized_quant_gb300 import workloads as W
        self.W, self.w = W, w
        L, U = w.num_layers, w.batch * w.num_kv_heads
        ncpu = os.cpu_count() or 1
        self.procs = max(1, min(procs or ncpu, L))
        n_s = self.procs
        self.layers = sorted({(i * L) // n_s for i in range(n_s)})
        self.n_s = len(self.layers)
        self.fraction = self.n_s / (L * U)
        self.S = w.context if prefill is None else prefill
        self.unit_w = W.scaled(w, batch=1, num_kv_heads=1, num_q_heads=w.num_q_heads // w.num_kv_heads)
        per = [[] for _ in range(self.procs)]
        self.owner = []
        for i, l in enumerate(self.layers):
            kb, vb, R, km, rpc = W.spec_fields(w.layers[l])
            k, v = W.gen_kv(self.unit_w, l, 0, self.S)
            per[i % self.procs].append((w.head_dim, w.group_size, kb, vb, R, km, rpc, k.numpy(), v.numpy()))
            self.owner.append(i % self.procs)
        self.per = [[i for i in range(self.n_s) if self.owner[i] == p] for p in range(self.procs)]
        # spawned workers, single-threaded numpy (a forked child of a CUDA
        # process can hang; spawn starts clean)
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.conns, self.workers = [], []
            for pidx in range(self.procs):
                a, b = ctx.Pipe()
                pr = ctx.Process(target=_oracle_worker, args=(b, per[pidx]), daemon=True)
                pr.start()
                self.conns.append(a)
                self.workers.append(pr)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for c in self.conns:
            if c.recv() != "ready":
                raise RuntimeError("oracle worker failed to start")
        self.pos = 0
        self.desc = (f"oracle decode step (append 1 token, then fp64 attention over the dequantized cache) on "
                     f"{self.n_s} of the step's {L * U} (layer, unit) pairs (layers {self.layers}, one unit each, "
                     f"prefill {self.S}), spread over {self.procs} worker processes of one host core each; "
                     f"tokens/s = batch x {self.n_s}/{L * U} / sample-step wall time")

    def step(self) -> float:
        """Wall seconds of one sample step (inputs drawn before the clock starts)."""
        msgs = [[] for _ in range(self.procs)]
        for i, l in enumerate(self.layers):
            k1, v1 = self.W.gen_kv(self.unit_w, l, self.S + self.pos, 1)
            q = self.W.gen_q(self.unit_w, l, self.pos).numpy()
            msgs[self.owner[i]].append((k1.numpy(), v1.numpy(), q))
        t0 = time.perf_counter()
        for c, m in zip(self.conns, msgs):
            c.send(m)
        for c in self.conns:
            if c.recv() != "done":
                raise RuntimeError("oracle worker failed")
        dt = time.perf_counter() - t0
        self.pos += 1
        return dt

    def tokens_per_s(self, seconds_per_step: float) -> float:
        return self.w.batch * self.fraction / seconds_per_step

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except Exception:
                pass
        for pr in self.workers:
            pr.join(timeout=10)
            if pr.is_alive():
                pr.terminate()


def quant_errors(w):
    """Quantization error of each distinct precision pair on one (batch, kv
    head) unit at full context (KVTuner A3's metrics): e_k, e_v over the
    quantized tokens, e_a = mean |a - a_hat| of the attention weights and e_o
    of the output for the first query, against fp64 over the fp16 K and V."""
    import numpy as np
    from mixed_precision_quantized_quant_gb300 import workloads as W
    from oracle import kvq_oracle as O
    unit_w = W.scaled(w, batch=1, num_kv_heads=1, num_q_heads=w.num_q_heads // w.num_kv_heads)
    out, seen = {}, set()
    for l, spec in enumerate(w.layers):
        if spec in seen:
            continue
        seen.add(spec)
        kb, vb, R, km, rpc = W.spec_fields(spec)
        ora = O.OracleLayerCache(1, 1, w.head_dim, w.group_size, kb, vb, R, km, rpc)
        k16, v16 = W.gen_kv(unit_w, l, 0, w.context)
        ora.append(k16.numpy(), v16.numpy())
        kh, vh = ora.dequantized(0)
        k, v = (x.numpy()[0, 0].astype(np.float64) for x in (k16, v16))
        q = W.gen_q(unit_w, l, 0).numpy()[0].astype(np.float64)
        ea, o_ref, o_hat = [], [], []
        for h in range(q.shape[0]):
            def weights(kk):
                x = kk @ q[h] / np.sqrt(kk.shape[1])
                e = np.exp(x - x.max())
                return e / e.sum()
            ea.append(np.abs(weights(k) - weights(kh)).mean())
            o_ref.append(O.attention_fp64(q[h], k, v))
            o_hat.append(O.attention_fp64(q[h], kh, vh))
        nq = ora.n_q
        out[f"K{kb}V{vb}"] = {"e_k": round(O.rel_error(k[:nq], kh[:nq]), 5),
                              "e_v": round(O.rel_error(v[:nq], vh[:nq]), 5),
                              "e_a": float(f"{np.mean(ea):.3e}"),
                              "e_o": round(O.rel_error(np.stack(o_ref), np.stack(o_hat)), 5)}
    return out


def oracle_sample(w, budget_s: float = 20.0, prefill=None):
    """(tokens/s, median seconds per sample step, cores, description) from
    sample steps repeated until about budget_s seconds of oracle work."""
    smp = OracleSampler(w, prefill=prefill)
    try:
        t_start = time.perf_counter()
        steps = []
        while len(steps) < 3 or (time.perf_counter() - t_start < budget_s and len(steps) < 200):
            steps.append(smp.step())
        step_s = statistics.median(steps)
        return smp.tokens_per_s(step_s), step_s, smp.procs, smp.desc + f"; median over {len(steps)} sample steps"
    finally:
        smp.close()


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
    return W.scaled(w, name=w.name + "-per-token-keys",
                    layers=tuple((kb, vb, r, 1, rpc) for kb, vb, r, _, rpc in map(W.spec_fields, w.layers)))


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal: context for the measured-copy fraction


def _prefill_length(w, warm, steps):
    """Prefill length: the context, less an offset that puts a key-group flush
    on every layer at the middle timed step.  A step appends one token, so
    step k (1-based, warm-up included) brings the cache to prefill + k tokens;
    a layer whose window is a multiple of G flushes when that count is a
    multiple of G."""
    mid = warm + (steps + 1) // 2
    return w.context - (mid % w.group_size), mid


def measure_decode(w, args, dev, world, e2e=True):
    """One workload's decode step on this GPU: prefill, warm-up, the timed
    window (per-step CUDA events), the decode-only roofline replays and the
    end-to-end leg.  Returns a dict of figures."""
    import torch

    from mixed_precision_quantized_quant_gb300 import kvq as K
    from mixed_precision_quantized_quant_gb300 import workloads as W

    L, B, Hq, Hkv, D = w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    steps, warm = args.steps, args.warmup
    S0, mid = _prefill_length(w, warm, steps)
    cap = S0 + warm + steps
    stream = torch.cuda.Stream(device=dev)
    cache = K.KVQCache(w.layers, B, Hq, Hkv, D, w.group_size, cap, device=dev)

    # ---- prefill (timed per layer: append GB/s)
    prefill_ms, prefill_bytes = 0.0, 0
    with torch.cuda.stream(stream):
        for l in range(L):
            k, v = W.gen_kv(w, l, 0, S0, device=dev)
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
            k1, v1 = W.gen_kv(w, l, S0 + s, 1, device=dev)
            kin[s, l].copy_(k1)
            vin[s, l].copy_(v1)
            qin[s, l].copy_(W.gen_q(w, l, s, device=dev))
    outs = torch.empty((L, B, Hq, D), dtype=torch.float32, device=dev)
    # inputs are staged into fixed buffers so the step graph is captured once
    k_cur = torch.empty((L, B, Hkv, 1, D), dtype=torch.float16, device=dev)
    v_cur = torch.empty_like(k_cur)
    q_cur = torch.empty((L, B, Hq, D), dtype=torch.float16, device=dev)
    torch.cuda.synchronize()
    Ks, Vs = [k_cur[l] for l in range(L)], [v_cur[l] for l in range(L)]
    Qs, Os = [q_cur[l] for l in range(L)], [outs[l] for l in range(L)]

    def run_step(s):
        k_cur.copy_(kin[s], non_blocking=True)
        v_cur.copy_(vin[s], non_blocking=True)
        q_cur.copy_(qin[s], non_blocking=True)
        cache.decode_step(Ks, Vs, Qs, Os, stream=stream)

    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    # The timed window (steps warm .. warm+steps-1) runs args.reps times: the
    # cache state after the warm-up is saved once (kvq_state_save) and restored
    # before every repetition, so each one decodes the same tokens from the
    # same state, flush step included.
    win_reps = max(10, args.reps)
    win_ms, step_rows = [], []
    with torch.cuda.stream(stream):
        for s in range(warm):
            run_step(s)
        snapshot = cache.save_state(stream=stream)
        stream.synchronize()
        nq_before = [cache.view(l)["quantized_tokens"] for l in range(L)]
        bytes_first = sum(cache.decode_bytes(l) for l in range(L))
        for r in range(win_reps):
            if r:
                cache.restore_state(snapshot, stream=stream)
            stream.synchronize()
            _barrier(world)
            torch.cuda.synchronize()
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
            t0 = time.time()
            evs[0].record(stream)
            for i, s in enumerate(range(warm, warm + steps)):
                run_step(s)
                evs[i + 1].record(stream)
            stream.synchronize()
            t1 = time.time()
            sampler.mark(t0, t1)
            torch.cuda.synchronize()
            _barrier(world)
            win_ms.append(_max_over_ranks(evs[0].elapsed_time(evs[-1]), world))
            step_rows.append([evs[i].elapsed_time(evs[i + 1]) for i in range(steps)])
        bytes_last = sum(cache.decode_bytes(l) for l in range(L))
        flushed = sum(1 for l in range(L) if cache.view(l)["quantized_tokens"] > nq_before[l])
        del snapshot
    ms_total = statistics.median(win_ms)
    # per step position: the median over the repetitions
    step_ms = [statistics.median(row[i] for row in step_rows) for i in range(steps)]
    ms_step = ms_total / steps
    flush_i = mid - warm - 1  # 0-based index of the flush step inside the window
    others = [t for i, t in enumerate(step_ms) if i != flush_i] or step_ms

    # ---- decode-attention roofline: replays of a decode-only graph of all
    # layers, one CUDA event pair per replay, median replay
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
        reps = max(10, min(100, int(100 / max(ms_step, 0.05))))
        rev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        t0 = time.time()
        rev[0].record(stream)
        for r in range(reps):
            g.replay()
            rev[r + 1].record(stream)
        stream.synchronize()
        sampler.mark(t0, time.time())
    replay_ms = sorted(rev[r].elapsed_time(rev[r + 1]) for r in range(reps))
    dec_ms_per_launch = statistics.median(replay_ms) / L
    dec_bytes_per_launch = sum(dec_bytes) / L
    clocks = sampler.stop()
    err = cache.device_error(stream)
    if err:
        raise RuntimeError(f"device error word {err}")
    res = {
        "w": w, "steps": steps, "warmup": warm, "ms_total": ms_total, "ms_step": ms_step,
        "tokens_per_s": world * B * steps / (ms_total / 1e3),
        "window_ms": {"median": round(ms_total, 4), "min": round(min(win_ms), 4), "max": round(max(win_ms), 4),
                      "repetitions": win_reps},
        "step_ms": {"median": round(statistics.median(step_ms), 4), "mean": round(ms_step, 4),
                    "flush_step": round(step_ms[flush_i], 4) if 0 <= flush_i < steps else None,
                    "median_without_flush_step": round(statistics.median(others), 4),
                    "min": round(min(step_ms), 4), "max": round(max(step_ms), 4),
                    "flush_step_index": flush_i, "layers_flushed_in_window": flushed},
        "prefill": S0, "bytes_step": (bytes_first + bytes_last) / 2,
        "append_gbs": prefill_bytes / (prefill_ms / 1e3) / 1e9,
        "dec_ms_per_launch": dec_ms_per_launch, "dec_bytes_per_launch": dec_bytes_per_launch,
        "replays": reps, "clocks": clocks, "equivalent_bits": cache.equivalent_bits(),
    }
    del kin, vin, qin, g

    # ---- end to end through the public API, pinned host copies every step
    res["e2e_tps"] = None
    res["h2d"] = L * (2 * B * Hkv * D * 2 + B * Hq * D * 2)
    res["d2h"] = L * B * Hq * D * 4
    if e2e:
        cache.close()
        del cache
        torch.cuda.empty_cache()
        h_k = torch.empty((nst, L, B, Hkv, 1, D), dtype=torch.float16).pin_memory()
        h_v = torch.empty_like(h_k).pin_memory()
        h_q = torch.empty((nst, L, B, Hq, D), dtype=torch.float16).pin_memory()
        for s in range(nst):
            for l in range(L):
                k1, v1 = W.gen_kv(w, l, S0 + s, 1, device=dev)
                h_k[s, l].copy_(k1)
                h_v[s, l].copy_(v1)
                h_q[s, l].copy_(W.gen_q(w, l, s, device=dev))
        h_out = torch.empty((2, L, B, Hq, D), dtype=torch.float32).pin_memory()  # two readback slots
        e2e_cache = K.KVQCache(w.layers, B, Hq, Hkv, D, w.group_size, cap, device=dev)
        with torch.cuda.stream(stream):
            for l in range(L):
                k, v = W.gen_kv(w, l, 0, S0, device=dev)
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
        e2e_snap = e2e_cache.save_state(stream=stream)
        e2e_win = []
        for r in range(win_reps):
            if r:
                e2e_cache.restore_state(e2e_snap, stream=stream)
            stream.synchronize()
            _barrier(world)
            t0 = time.perf_counter()
            run(warm, steps)
            t1 = time.perf_counter()
            _barrier(world)
            e2e_win.append(_max_over_ranks(t1 - t0, world))
        del e2e_snap
        e2e_s = statistics.median(e2e_win)
        res["e2e_tps"] = world * B * steps / e2e_s
        res["e2e_window_s"] = {"median": round(e2e_s, 5), "min": round(min(e2e_win), 5),
                               "max": round(max(e2e_win), 5), "repetitions": win_reps}
        if e2e_cache.device_error(stream):
            raise RuntimeError("device error word set (end-to-end leg)")
        e2e_cache.close()
    else:
        cache.close()
    torch.cuda.empty_cache()
    return res


def run_gpu(args):
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
    m = measure_decode(w, args, dev, world, e2e=not args.no_e2e)

    peak, peak_kind = _peaks()
    achieved = m["dec_bytes_per_launch"] / (m["dec_ms_per_launch"] / 1e3) / 1e9
    # the committed capture covers every layer of the workload: no figure for a layer subset
    traffic = None if args.layers else _ncu_traffic(w.name)
    L = w.num_layers
    bytes_step = m["bytes_step"]
    result = {
        "metric": METRIC,
        "value": round(m["tokens_per_s"], 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": m["steps"],
        "warmup": m["warmup"],
        "ms_per_step": round(m["ms_step"], 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 codes/fp32 accumulate",
        "data": "synthetic (seeded: keys N(mu_c, sigma_c) with channel outliers, values with drifting mean)",
        "config": {**w.describe(), "prefill": m["prefill"], "equivalent_bits": round(m["equivalent_bits"], 5),
                   "parallelism": f"replicas x{world} (independent (batch, kv head) units, no collective)",
                   "window": (f"steps {m['warmup'] + 1}..{m['warmup'] + m['steps']} after a {m['prefill']}-token "
                              f"prefill; step {m['warmup'] + m['step_ms']['flush_step_index'] + 1} brings every "
                              f"layer to a multiple of G tokens and flushes a key group (quantize + pack)"),
                   "l2": ("inputs larger than L2: %.2f GB of cache read per step" % (bytes_step / 1e9)
                          if bytes_step > L2_BYTES else
                          "cache smaller than L2 (%.3f MB read per step), not flushed: a latency figure"
                          % (bytes_step / 1e6))},
        "step_ms": m["step_ms"],
        "window_ms": m["window_ms"],
        "cache_read_gbs": round(bytes_step / (m["ms_step"] / 1e3) / 1e9, 1),
        "cache_read_frac_of_peak": round(bytes_step / (m["ms_step"] / 1e3) / 1e9 / peak, 4),
        "append_prefill_gbs": round(m["append_gbs"], 1),
        "append_prefill_frac_of_peak": round(m["append_gbs"] / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "kernel": "decode_kernel (all layers, decode-only graph replay, median of "
                               f"{m['replays']} replays)",
                     "bytes_per_launch": int(m["dec_bytes_per_launch"]),
                     "us_per_launch": round(m["dec_ms_per_launch"] * 1e3, 3),
                     "peak_source": f"{peak_kind} HBM copy bandwidth (frac); frac_of_nominal against the "
                                    f"{NOMINAL_HBM_GBS:.0f} GB/s HBM3e nominal"},
        "e2e": None if m["e2e_tps"] is None else {"value": round(m["e2e_tps"], 1), "unit": "tokens/s",
                                                  "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"],
                                                  "window_s": m["e2e_window_s"]},
        "gpu_launches": m["steps"] * 2 * L,
        "timing": (f"median of {m['window_ms']['repetitions']} repetitions of the {m['steps']}-step window, each "
                   "from the cache state saved after the warm-up (kvq_state_save / kvq_state_restore); "
                   "gpu_launches counts one window"),
        "clocks": m["clocks"],
    }
    # the other decode workloads, measured in the same run (no end-to-end leg)
    extra = {}
    if not args.layers:
        for idx in args.extra_workloads:
            if idx == args.workload:
                continue
            wx = _with_key_mode(W.workload(idx), args)
            mx = measure_decode(wx, args, dev, world, e2e=False)
            ax = mx["dec_bytes_per_launch"] / (mx["dec_ms_per_launch"] / 1e3) / 1e9
            extra[wx.name] = {"tokens_per_s": round(mx["tokens_per_s"], 1), "ms_per_step": round(mx["ms_step"], 5),
                              "step_ms": mx["step_ms"], "prefill": mx["prefill"],
                              "decode_kernel_gbs": round(ax, 1), "decode_kernel_frac": round(ax / peak, 4),
                              "append_prefill_gbs": round(mx["append_gbs"], 1),
                              "append_prefill_frac_of_peak": round(mx["append_gbs"] / peak, 4),
                              "clocks": mx["clocks"]}
    if extra:
        result["other_workloads"] = extra
    if not args.layers and not args.no_chunk:
        result["chunk_tflops"] = measure_chunk_layers(dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, step_s, cores, desc = oracle_sample(w, budget_s=args.cpu_budget, prefill=m["prefill"])
        result["cpu_baseline"] = {"value": round(tps, 6), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                  "sample": desc, "seconds_per_sample_step": round(step_s, 3)}
        result["quant_error"] = {"per_pair": quant_errors(w),
                                 "of": "one (batch, kv head) unit at full context, first query; e_k, e_v over "
                                       "its quantized tokens, e_a and e_o against fp64 attention over the fp16 "
                                       "K and V (KVTuner A3)"}
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
            kb, vb, R, km, rpc = W.spec_fields(w.layers[l])
            ora = O.OracleLayerCache(1, 1, D, w.group_size, kb, vb, R, km, rpc)
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


def measure_chunk_layers(dev, workload=2, layers=3, batch=2, reps=10):
    """Causal chunk attention (every query of the context over the layer's
    quantized cache) on the first `layers` layers of a workload at `batch`
    sequences: median over `reps` timed passes of the layers (CUDA events on
    the launching stream); TFLOP/s counts 4 d per visible (query, key) pair."""
    import torch

    from mixed_precision_quantized_quant_gb300 import kvq as K
    from mixed_precision_quantized_quant_gb300 import workloads as W

    w = W.scaled(W.workload(workload), batch=batch)
    w = W.scaled(w, num_layers=layers, layers=tuple(w.layers[:layers]))
    L, B, Hq, Hkv, D, T = w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.context
    stream = torch.cuda.Stream(device=dev)
    cache = K.KVQCache(w.layers, B, Hq, Hkv, D, w.group_size, T, device=dev)
    with torch.cuda.stream(stream):
        for l in range(L):
            k, v = W.gen_kv(w, l, 0, T, device=dev)
            cache.append(l, k, v, stream=stream)
            del k, v
        gen = torch.Generator(device=dev)
        gen.manual_seed(11)
        q = torch.randn((B, Hq, T, D), generator=gen, device=dev).half()
        out = torch.empty((B, Hq, T, D), dtype=torch.float32, device=dev)
        for _ in range(3):
            for l in range(L):
                cache.chunk_attn(l, q, out, stream=stream)
        stream.synchronize()
        ms = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for l in range(L):
                cache.chunk_attn(l, q, out, stream=stream)
            e1.record(stream)
            stream.synchronize()
            ms.append(e0.elapsed_time(e1))
    if cache.device_error(stream):
        raise RuntimeError("device error word set (chunk attention)")
    cache.close()
    med = statistics.median(ms)
    tflops = L * _chunk_flops(B, Hq, D, T, T) / (med / 1e3) / 1e12
    peak, kind = _tensor_peak()
    return {"value": round(tflops, 2), "unit": "TFLOP/s", "frac_of_bf16_peak": round(tflops / peak, 4),
            "peak": peak, "peak_source": f"{kind} bf16 dense",
            "config": {"workload": w.name, "layers": L, "batch": B, "queries": T, "context": T},
            "ms_per_pass": round(med, 4), "passes": reps,
            "kernel": "chunk_attn_kernel (tcgen05, accumulators in tensor memory) after its dequantize pass"}


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
    S0, _ = _prefill_length(w, args.warmup, args.steps)
    smp = OracleSampler(w, prefill=S0)
    try:
        for _ in range(args.warmup):
            smp.step()
        vals = [smp.step() for _ in range(args.steps)]
    finally:
        smp.close()
    total = sum(vals)
    step_s = total / args.steps
    v = smp.tokens_per_s(step_s)
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": round(v, 6), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 quantizer / f64 attention",
        "data": "synthetic (seeded: keys N(mu_c, sigma_c) with channel outliers, values with drifting mean)",
        "config": {**w.describe(), "prefill": S0},
        "cpu_baseline": {"value": round(v, 6), "unit": "tokens/s", "cores": smp.procs, "kind": "oracle",
                         "sample": smp.desc + f"; {args.steps} timed sample steps after {args.warmup} warm-up"},
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
    ap.add_argument("--workload", type=int, default=None,
                    help="1..6; decode default 5, the Llama-2-70B-shaped 32K-context decode (the largest); "
                         "chunk default 2, the Llama-3.1-8B-shaped prefill")
    ap.add_argument("--extra-workloads", type=lambda x: [int(t) for t in x.split(",") if t], default=[2],
                    help="comma-separated workloads measured after the main one and reported under "
                         "other_workloads (decode only; empty to skip)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--reps", type=int, default=10,
                    help="repetitions of the timed window (at least 10), each from the same saved cache state")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="profiling runs: skip the end-to-end leg")
    ap.add_argument("--no-chunk", action="store_true", help="skip the chunk-attention extra key")
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
    if args.workload is None:
        args.workload = 2 if args.op == "chunk" else 5
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
