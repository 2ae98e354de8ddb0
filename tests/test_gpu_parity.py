"""GPU parity: the CUDA path against the oracle, through the C ABI.

Packed codes, scales, zeros and the FP16 window are compared byte for byte;
attention outputs must be within max-abs 2e-3 and relative L2 1e-3 of fp64
attention over the same dequantized values."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import kvq_oracle as O
from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import workloads as W
from tests.kvq_testutil import assert_attn_close, compare_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    K.load()


def _rand_kv(gen, B, H, n, d, t0, total, outlier_ch=(3, 17), device="cuda"):
    k = torch.randn((B, H, n, d), generator=gen, device=device) * 1.5 + 0.3
    for c in outlier_ch:
        if c < d:
            k[..., c] *= 12.0
    m = 4.0 * (torch.arange(t0, t0 + n, device=device, dtype=torch.float32) / max(total - 1, 1))
    v = torch.randn((B, H, n, d), generator=gen, device=device) + m[None, None, :, None]
    return k.half().contiguous(), v.half().contiguous()


def _run_stream(kb, vb, D, G, R, gqa, schedule, B=2, Hkv=2, attn_every=1, seed=0, key_mode=0, rpc=0):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    total = sum(schedule)
    cache = K.KVQCache([(kb, vb, R, key_mode, rpc)], B, Hkv * gqa, Hkv, D, G, total)
    ora = O.OracleLayerCache(B, Hkv, D, G, kb, vb, R, key_mode, rpc)
    pos = 0
    for step, n in enumerate(schedule):
        k, v = _rand_kv(gen, B, Hkv, n, D, pos, total)
        cache.append(0, k, v)
        ora.append(k.cpu().numpy(), v.cpu().numpy())
        pos += n
        torch.cuda.synchronize()
        compare_layer(cache, 0, ora)
        assert cache.view(0)["window_bound"] == ora.bound
        if step % attn_every == 0 or step == len(schedule) - 1:
            q = torch.randn((B, Hkv * gqa, D), generator=gen, device="cuda").half()
            out = cache.decode_attn(0, q)
            torch.cuda.synchronize()
            exp = ora.attend(q.cpu().numpy())
            assert_attn_close(out.cpu().numpy(), exp, f"K{kb}V{vb} D{D} G{G} R{R} step {step} T={pos}")
    assert cache.device_error() == 0
    cache.close()


PAIRS = [(kb, vb) for kb in (2, 3, 4, 8) for vb in (2, 3, 4, 8)]


@pytest.mark.parametrize("kb,vb", PAIRS)
@pytest.mark.parametrize("D", [64, 128])
def test_stream_bitexact_and_attention(kb, vb, D):
    # R != G; a ragged prefill, decode steps across two flushes, a multi-token
    # chunk whose flush straddles the window and the input
    sched = [150] + [1] * 40 + [45, 1, 1, 77]
    _run_stream(kb, vb, D, 32, 64, 4, sched, attn_every=5)


@pytest.mark.parametrize("kb", [2, 4, 8])
@pytest.mark.parametrize("vb", [2, 3, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_per_token_keys_bitexact_and_attention(kb, vb, D):
    # KVTuner's per-token-asym key mode: same stream schedule, keys quantized per token
    sched = [150] + [1] * 40 + [45, 1, 1, 77]
    _run_stream(kb, vb, D, 32, 64, 4, sched, attn_every=5, seed=kb * 16 + vb, key_mode=K.KEY_PER_TOKEN)


@pytest.mark.parametrize("gqa", [1, 5, 8])
@pytest.mark.parametrize("G", [64, 128])
def test_per_token_keys_gqa_and_group_sizes(gqa, G):
    _run_stream(4, 2, 128, G, G, gqa, [3 * G + 5] + [1] * (G + 2), attn_every=9, seed=gqa + G,
                key_mode=K.KEY_PER_TOKEN)


@pytest.mark.parametrize("kb,vb", [(4, 2), (8, 4), (4, 8), (8, 8), (2, 4)])
@pytest.mark.parametrize("gqa", [5, 8])
def test_eight_head_tiles_group_128(kb, vb, gqa):
    # 5-8 query heads per kv head at G = 128: the transposed 8-head form, whose
    # four warps take the four 32-token slices of one key group per stage; a
    # ragged prefill, then decode steps through a flush
    _run_stream(kb, vb, 128, 128, 128, gqa, [3 * 128 + 5] + [1] * 130, attn_every=9, seed=kb * 16 + vb + gqa)


@pytest.mark.parametrize("kb,vb,D,key_mode", [(4, 2, 64, 0), (8, 8, 64, 0), (2, 4, 64, 0), (8, 4, 64, 1),
                                              (3, 4, 128, 0), (4, 3, 64, 0)])
def test_append_group_128_cta_forms(kb, vb, D, key_mode):
    # G = 128 flushes run 256-thread single-stage CTAs without 3-bit codes and
    # 512-thread double-stage CTAs with them: head_dim 64 for the first form
    # (value scales on the threads after the 64 channel ones), 3-bit pairs for
    # the second; a ragged prefill, then decode steps through a flush
    _run_stream(kb, vb, D, 128, 128, 4, [3 * 128 + 5] + [1] * 130, attn_every=13, seed=kb * 16 + vb + D,
                key_mode=key_mode)


@pytest.mark.parametrize("gqa", [1, 2, 3, 4, 5, 7, 8])
def test_gqa_ratios(gqa):
    _run_stream(4, 2, 128, 32, 32, gqa, [96 + 17] + [1] * 20, attn_every=4, seed=gqa)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_group_sizes_flush_boundaries(G):
    # prefill lengths = 0, 1, G-1 and G (mod G) around the window
    for n0 in (G, G + 1, 2 * G - 1, 3 * G):
        _run_stream(4, 4, 128, G, G, 4, [n0] + [1] * (G + 2), attn_every=7, seed=n0)


@pytest.mark.parametrize("kb,vb,key_mode", [(4, 3, 0), (2, 2, 0), (3, 4, 0), (8, 4, 1)])
@pytest.mark.parametrize("D", [64, 128])
def test_rpc_dynamic_window_stream(kb, vb, key_mode, D):
    # KVmix's shrinking window: R = 160 at 20%, a prefill that leaves 140 window
    # tokens, then decode steps: the 20th brings the window to 160, the bound
    # becomes 32 and five groups are quantized in that one step; later steps
    # flush one group every 32.  A 45-token chunk keeps the bound.  Records,
    # window, bound and attention against the oracle after every call.
    sched = [300] + [1] * 19 + [1] + [1] * 40 + [45] + [1] * 30
    _run_stream(kb, vb, D, 32, 160, 4, sched, attn_every=3, seed=kb * 16 + vb + D, key_mode=key_mode, rpc=20)


@pytest.mark.parametrize("G,R,rpc", [(64, 320, 10), (128, 640, 20), (32, 800, 20)])
def test_rpc_group_sizes(G, R, rpc):
    # shrinks at other group sizes and ratios; a prefill shorter than the
    # window first, so the first flushes come from decode steps alone
    sched = [R - 3] + [1] * (2 * G + 7)
    _run_stream(4, 2, 128, G, R, 8, sched, attn_every=11, seed=G + rpc, rpc=rpc)


def test_prefill_shorter_than_window():
    _run_stream(4, 2, 128, 32, 128, 4, [50, 1, 1, 1], attn_every=1)


def test_single_token_and_empty():
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    cache = K.KVQCache([(4, 2, 32)], 1, 8, 2, 64, 32, 64)
    q = torch.randn((1, 8, 64), generator=gen, device="cuda").half()
    with pytest.raises(K.KVQError) as ei:
        cache.decode_attn(0, q)
    assert ei.value.status == 6  # KVQ_ERR_STATE
    k, v = _rand_kv(gen, 1, 2, 1, 64, 0, 1)
    cache.append(0, k, v)
    out = cache.decode_attn(0, q).cpu().numpy()
    # one token: the output of every query head is that token's value
    vv = v.cpu().numpy().astype(np.float64)
    for h in range(8):
        assert np.allclose(out[0, h], vv[0, h // 4, 0], atol=1e-6)
    cache.close()


def test_capacity_and_argument_errors():
    cache = K.KVQCache([(4, 2, 32)], 1, 4, 1, 128, 32, 40)
    k = torch.zeros((1, 1, 41, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(K.KVQError) as ei:
        cache.append(0, k, k)
    assert ei.value.status == 4
    with pytest.raises(K.KVQError) as ei:
        K.kvq_append(cache.h, 1, int(k.data_ptr()), int(k.data_ptr()), 1, 0)
    assert ei.value.status == 1
    with pytest.raises(K.KVQError) as ei:
        K.kvq_append(cache.h, 0, int(k.data_ptr()) + 2, int(k.data_ptr()), 1, 0)
    assert ei.value.status == 3
    assert cache.view(0)["tokens"] == 0
    cache.close()


@pytest.mark.parametrize("layers", [((8, 4, 32), (4, 2, 32), (2, 2, 64)),
                                    ((8, 4, 32, 1), (4, 2, 32, 0), (4, 4, 64, 1)),
                                    ((4, 3, 160, 0, 20), (2, 2, 96, 0, 10), (8, 4, 32))])
def test_decode_step_graph_matches_layer_calls(layers):
    w = W.scaled(W.workload(2), batch=2, num_layers=3, context=200, decode_steps=40, layers=layers)
    stream = torch.cuda.Stream()
    caches = []
    for _ in range(2):
        c = K.KVQCache(w.layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size,
                       w.total_tokens)
        for l in range(w.num_layers):
            k, v = W.gen_kv(w, l, 0, w.context, device="cuda")
            c.append(l, k, v)
        caches.append(c)
    torch.cuda.synchronize()
    outs_a = [torch.empty((w.batch, w.num_q_heads, w.head_dim), device="cuda") for _ in range(w.num_layers)]
    outs_b = [torch.empty_like(o) for o in outs_a]
    for step in range(35):
        ks, vs, qs = [], [], []
        for l in range(w.num_layers):
            k, v = W.gen_kv(w, l, w.context + step, 1, device="cuda")
            ks.append(k)
            vs.append(v)
            qs.append(W.gen_q(w, l, step, device="cuda"))
        with torch.cuda.stream(stream):
            caches[0].decode_step(ks, vs, qs, outs_a, stream=stream)
            for l in range(w.num_layers):
                caches[1].append(l, ks[l], vs[l], stream=stream)
                caches[1].decode_attn(l, qs[l], outs_b[l], stream=stream)
        stream.synchronize()
        for l in range(w.num_layers):
            assert torch.equal(outs_a[l], outs_b[l]), (step, l)
            va, vb = caches[0].view(l), caches[1].view(l)
            assert [va[k] for k in ("tokens", "quantized_tokens", "window_bound")] == \
                [vb[k] for k in ("tokens", "quantized_tokens", "window_bound")], (step, l)
    for c in caches:
        assert c.device_error() == 0
        c.close()



def test_decode_step_graph_replay_fixed_buffers():
    """The step graph captured once and replayed with the same input and
    output buffers every step (the launch configuration the benchmark times:
    every decode a programmatic dependent of the previous layer's), bit for
    bit against per-layer calls, across group flushes."""
    layers = ((8, 4, 32), (4, 2, 32), (4, 2, 32), (2, 2, 64))
    w = W.scaled(W.workload(2), batch=3, num_layers=4, context=190, decode_steps=80, layers=layers)
    L = w.num_layers
    stream = torch.cuda.Stream()
    caches = []
    for _ in range(2):
        c = K.KVQCache(w.layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size,
                       w.total_tokens)
        for l in range(L):
            k, v = W.gen_kv(w, l, 0, w.context, device="cuda")
            c.append(l, k, v)
        caches.append(c)
    k_cur = torch.empty((L, w.batch, w.num_kv_heads, 1, w.head_dim), dtype=torch.float16, device="cuda")
    v_cur = torch.empty_like(k_cur)
    q_cur = torch.empty((L, w.batch, w.num_q_heads, w.head_dim), dtype=torch.float16, device="cuda")
    outs_a = torch.empty((L, w.batch, w.num_q_heads, w.head_dim), device="cuda")
    outs_b = torch.empty_like(outs_a)
    torch.cuda.synchronize()
    for step in range(70):
        for l in range(L):
            k, v = W.gen_kv(w, l, w.context + step, 1, device="cuda")
            k_cur[l].copy_(k)
            v_cur[l].copy_(v)
            q_cur[l].copy_(W.gen_q(w, l, step, device="cuda"))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            caches[0].decode_step([k_cur[l] for l in range(L)], [v_cur[l] for l in range(L)],
                                  [q_cur[l] for l in range(L)], [outs_a[l] for l in range(L)], stream=stream)
            for l in range(L):
                caches[1].append(l, k_cur[l], v_cur[l], stream=stream)
                caches[1].decode_attn(l, q_cur[l], outs_b[l], stream=stream)
        stream.synchronize()
        assert torch.equal(outs_a, outs_b), step
    for c in caches:
        assert c.device_error() == 0
        c.close()

def _unit_stream(k, v, u, Hkv):
    b, h = divmod(u, Hkv)
    return k[b:b + 1, h:h + 1].cpu().numpy(), v[b:b + 1, h:h + 1].cpu().numpy()


@pytest.mark.parametrize("idx", [1])
def test_workload_tiny_every_step(idx):
    w = W.workload(idx)
    cache = K.KVQCache(w.layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size,
                       w.total_tokens)
    kb, vb, R = w.layers[0][:3]
    ora = O.OracleLayerCache(w.batch, w.num_kv_heads, w.head_dim, w.group_size, kb, vb, R)
    k, v = W.gen_kv(w, 0, 0, w.context, device="cuda")
    cache.append(0, k, v)
    ora.append(k.cpu().numpy(), v.cpu().numpy())
    for step in range(w.decode_steps):
        k, v = W.gen_kv(w, 0, w.context + step, 1, device="cuda")
        q = W.gen_q(w, 0, step, device="cuda")
        cache.append(0, k, v)
        out = cache.decode_attn(0, q)
        ora.append(k.cpu().numpy(), v.cpu().numpy())
        torch.cuda.synchronize()
        compare_layer(cache, 0, ora)
        assert_attn_close(out.cpu().numpy(), ora.attend(q.cpu().numpy()), f"step {step}")
    assert cache.device_error() == 0
    cache.close()


def _layers_to_check(w):
    """One layer of every distinct (k_bits, v_bits, R) in the table."""
    seen, out = set(), []
    for l, p in enumerate(w.layers):
        if p not in seen:
            seen.add(p)
            out.append(l)
    return out


@pytest.mark.parametrize("idx,key_mode", [(2, 0), (3, 0), (4, 0), (5, 0), (3, 1), (6, 0)])
def test_workload_full_size_sampled(idx, key_mode):
    """Full-size shapes in the benchmark's launch configuration, one layer per
    distinct precision pair; codes and attention checked on sampled units.
    (3, 1): the Qwen2.5-7B-shaped workload with every layer in the
    per-token-asym key mode, the mode KVTuner pairs with that model;
    6: the KVmix page's own K3V4 orientation.)"""
    w = W.workload(idx)
    if key_mode:
        w = W.scaled(w, layers=tuple((kb, vb, r, key_mode, rpc) for kb, vb, r, _, rpc in map(W.spec_fields, w.layers)))
    layers = _layers_to_check(w)
    steps = min(w.decode_steps, 40)
    sub = [w.layers[l] for l in layers]
    cache = K.KVQCache(sub, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size,
                       w.context + steps)
    U = w.batch * w.num_kv_heads
    units = sorted({0, U - 1, U // 2, (U * 7) // 11})
    rep = w.num_q_heads // w.num_kv_heads
    for li, l in enumerate(layers):
        kb, vb, R, km, rpc = W.spec_fields(w.layers[l])
        k, v = W.gen_kv(w, l, 0, w.context, device="cuda")
        cache.append(li, k, v)
        oras = {}
        for u in units:
            o = O.OracleLayerCache(1, 1, w.head_dim, w.group_size, kb, vb, R, km, rpc)
            o.append(*_unit_stream(k, v, u, w.num_kv_heads))
            oras[u] = o
        del k, v
        check_steps = {0, 1, steps - 1} | {s for s in range(steps)
                                           if (w.context + s + 1 - R) % w.group_size == 0}
        for s in range(steps):
            k1, v1 = W.gen_kv(w, l, w.context + s, 1, device="cuda")
            q = W.gen_q(w, l, s, device="cuda")
            cache.append(li, k1, v1)
            out = cache.decode_attn(li, q)
            for u in units:
                oras[u].append(*_unit_stream(k1, v1, u, w.num_kv_heads))
            if s in check_steps:
                torch.cuda.synchronize()
                outn = out.cpu().numpy()
                qn = q.cpu().numpy()
                for u in units:
                    b, h = divmod(u, w.num_kv_heads)
                    _check_unit(cache, li, u, oras[u])
                    exp = oras[u].attend(qn[b:b + 1, h * rep:(h + 1) * rep])
                    assert_attn_close(outn[b, h * rep:(h + 1) * rep], exp[0],
                                      f"workload {idx} layer {l} step {s} unit {u}")
    assert cache.device_error() == 0
    cache.close()


def _check_unit(cache, layer, u, ora):
    from tests.kvq_testutil import gpu_unit_records, gpu_unit_ring
    got = gpu_unit_records(cache, layer, u)
    assert got == ora.unit_records(0), f"records unit {u}"
    live = ora.live_ring_slots()
    if len(live):
        gk, gv = gpu_unit_ring(cache, layer, u)
        ok_, ov_ = ora.residual_ring(0)
        assert np.array_equal(gk[live].view(np.uint16), ok_[live].view(np.uint16))
        assert np.array_equal(gv[live].view(np.uint16), ov_[live].view(np.uint16))
