"""GPU parity of the causal chunk attention (tcgen05 kernel) against the
oracle, through the C ABI: queries of the n newest tokens over the cache as
it stands (KVTuner A2 calibration: prefill over the dequantized cache).
Outputs must be within max-abs 2e-3 and relative L2 1e-3 of fp64 attention
over the same dequantized values."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import kvq_oracle as O
from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import workloads as W
from tests.kvq_testutil import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    K.load()


def _kv(gen, B, H, n, d, t0, total):
    # channel-outlier keys and drifting values, as in the decode parity tests
    k = torch.randn((B, H, n, d), generator=gen, device="cuda") * 1.5 + 0.3
    for c in (3, 17, 40):
        if c < d:
            k[..., c] *= 12.0
    m = 4.0 * (torch.arange(t0, t0 + n, device="cuda", dtype=torch.float32) / max(total - 1, 1))
    v = torch.randn((B, H, n, d), generator=gen, device="cuda") + m[None, None, :, None]
    return k.half().contiguous(), v.half().contiguous()


def _case(kb, vb, D, G, R, gqa, appends, chunks, B=2, Hkv=2, key_mode=0, seed=0):
    """Append `appends` token counts, then check chunk attention for each n in
    `chunks` (n queries of the newest tokens) against the oracle."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    T = sum(appends)
    Hq = Hkv * gqa
    cache = K.KVQCache([(kb, vb, R, key_mode)], B, Hq, Hkv, D, G, T)
    ora = O.OracleLayerCache(B, Hkv, D, G, kb, vb, R, key_mode)
    pos = 0
    for n in appends:
        k, v = _kv(gen, B, Hkv, n, D, pos, T)
        cache.append(0, k, v)
        ora.append(k.cpu().numpy(), v.cpu().numpy())
        pos += n
    for n in chunks:
        q = torch.randn((B, Hq, n, D), generator=gen, device="cuda").half()
        out = cache.chunk_attn(0, q)
        torch.cuda.synchronize()
        exp = ora.attend_chunk(q.cpu().numpy())
        assert_attn_close(out.cpu().numpy(), exp, f"K{kb}V{vb} D{D} G{G} R{R} gqa{gqa} T={T} n={n} km{key_mode}")
    assert cache.device_error() == 0
    cache.close()


PAIRS = [(kb, vb) for kb in (2, 3, 4, 8) for vb in (2, 3, 4, 8)]


@pytest.mark.parametrize("kb,vb", PAIRS)
def test_chunk_all_pairs_d128(kb, vb):
    # full causal prefill (n = T) and a chunk that starts inside the quantized part
    _case(kb, vb, 128, 32, 32, 4, [137, 63], [200, 45, 1])


@pytest.mark.parametrize("kb,vb", [(2, 2), (3, 4), (4, 3), (8, 8)])
def test_chunk_pairs_d64(kb, vb):
    _case(kb, vb, 64, 32, 64, 4, [250], [250, 77])


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 2), (8, 4), (4, 8)])
def test_chunk_per_token_keys(kb, vb):
    _case(kb, vb, 128, 32, 32, 4, [190], [190, 33], key_mode=K.KEY_PER_TOKEN)


@pytest.mark.parametrize("gqa,G,R", [(1, 64, 64), (7, 32, 96), (8, 128, 128), (5, 64, 256), (2, 32, 32)])
def test_chunk_gqa_groups_windows(gqa, G, R):
    # gqa 7 and 5 leave rows of the 128-row tile unused; gqa 1 puts 128 queries in a tile
    _case(4, 2, 128, G, R, gqa, [3 * G + 41, 20], [3 * G + 61, 64, 2])


def test_chunk_window_only():
    # window longer than the context: nothing is quantized
    _case(3, 3, 128, 32, 256, 4, [100, 30], [130, 7])


def test_chunk_one_query_matches_decode():
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    B, Hkv, gqa, D, T = 2, 2, 4, 128, 333
    cache = K.KVQCache([(4, 2, 64)], B, Hkv * gqa, Hkv, D, 32, T)
    k, v = _kv(gen, B, Hkv, T, D, 0, T)
    cache.append(0, k, v)
    q = torch.randn((B, Hkv * gqa, D), generator=gen, device="cuda").half()
    dec = cache.decode_attn(0, q)
    chk = cache.chunk_attn(0, q[:, :, None, :].contiguous())[:, :, 0, :]
    torch.cuda.synchronize()
    diff = (dec - chk).abs().max().item()
    assert diff <= 2e-3, diff
    cache.close()


def test_chunk_argument_errors():
    cache = K.KVQCache([(4, 2, 32)], 1, 4, 1, 64, 32, 64)
    q = torch.zeros((1, 4, 1, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(K.KVQError) as e:
        cache.chunk_attn(0, q)
    assert e.value.status == 6  # empty layer
    k = torch.zeros((1, 1, 10, 64), dtype=torch.float16, device="cuda")
    cache.append(0, k, k)
    with pytest.raises(K.KVQError) as e:
        cache.chunk_attn(0, torch.zeros((1, 4, 11, 64), dtype=torch.float16, device="cuda"))
    assert e.value.status == 1  # more queries than tokens
    ws = torch.empty(K.kvq_chunk_workspace_bytes(cache.h), dtype=torch.uint8, device="cuda")
    with pytest.raises(K.KVQError) as e:
        K.kvq_chunk_attn(cache.h, 0, int(q.data_ptr()), 0, int(q.data_ptr()), int(ws.data_ptr()), ws.numel(), 0)
    assert e.value.status == 1
    with pytest.raises(K.KVQError) as e:  # workspace one byte short
        K.kvq_chunk_attn(cache.h, 0, int(q.data_ptr()), 1, int(q.data_ptr()), int(ws.data_ptr()), ws.numel() - 1, 0)
    assert e.value.status == 4
    assert cache.device_error() == 0
    cache.close()


@pytest.mark.parametrize("kb,vb", [(8, 4), (4, 2)])
def test_chunk_full_size_prefill_sampled(kb, vb):
    """Llama-3.1-8B-shaped causal prefill over the quantized cache: 4096
    tokens, 8 kv heads, 32 query heads, d128, G = R = 32, all queries at once.
    Rows are checked for sampled (unit, query) pairs against fp64 attention
    over the oracle's dequantized unit."""
    w = W.scaled(W.workload(2), batch=2, decode_steps=1)
    T, D, Hkv, Hq = w.context, w.head_dim, w.num_kv_heads, w.num_q_heads
    cache = K.KVQCache([(kb, vb, w.group_size)], w.batch, Hq, Hkv, D, w.group_size, T)
    k, v = W.gen_kv(w, 0, 0, T, device="cuda")
    cache.append(0, k, v)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    q = torch.randn((w.batch, Hq, T, D), generator=gen, device="cuda").half()
    out = cache.chunk_attn(0, q)
    torch.cuda.synchronize()
    assert cache.device_error() == 0
    U = w.batch * Hkv
    rep = Hq // Hkv
    units = sorted({0, U - 1, U // 2 + 1})
    queries = [0, 1, 31, 32, 63, 64, 65, 1000, 2047, 2048, 4000, T - 1]
    kn, vn = k.cpu().numpy(), v.cpu().numpy()
    qn = q.cpu().numpy()
    on = out.cpu().numpy()
    for u in units:
        b, h = divmod(u, Hkv)
        ora = O.OracleLayerCache(1, 1, D, w.group_size, kb, vb, w.group_size)
        ora.append(kn[b:b + 1, h:h + 1], vn[b:b + 1, h:h + 1])
        kh, vh = ora.dequantized(0)
        got, exp = [], []
        for j in (0, rep - 1):
            for i in queries:
                exp.append(O.attention_fp64(qn[b, h * rep + j, i].astype(np.float64), kh[: i + 1], vh[: i + 1]))
                got.append(on[b, h * rep + j, i])
        assert_attn_close(np.stack(got), np.stack(exp), f"unit {u} K{kb}V{vb}")
    cache.close()


def test_chunk_after_single_token_appends():
    """Chunks of several sizes after each of a run of one-token appends, so
    the window fills, flushes and wraps between calls."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(21)
    B, Hkv, gqa, D, G, R = 1, 2, 4, 128, 32, 64
    T0, steps = 100, 45
    cache = K.KVQCache([(4, 3, R)], B, Hkv * gqa, Hkv, D, G, T0 + steps)
    ora = O.OracleLayerCache(B, Hkv, D, G, 4, 3, R)
    k, v = _kv(gen, B, Hkv, T0, D, 0, T0 + steps)
    cache.append(0, k, v)
    ora.append(k.cpu().numpy(), v.cpu().numpy())
    for s in range(steps):
        k, v = _kv(gen, B, Hkv, 1, D, T0 + s, T0 + steps)
        cache.append(0, k, v)
        ora.append(k.cpu().numpy(), v.cpu().numpy())
        if s % 7 == 0 or s == steps - 1:
            n = 1 + (s * 13) % 70
            q = torch.randn((B, Hkv * gqa, n, D), generator=gen, device="cuda").half()
            out = cache.chunk_attn(0, q)
            torch.cuda.synchronize()
            assert_attn_close(out.cpu().numpy(), ora.attend_chunk(q.cpu().numpy()), f"step {s} n {n}")
    assert cache.device_error() == 0
    cache.close()


@pytest.mark.parametrize("idx,key_mode,n", [(3, 1, 512), (4, 0, 256), (6, 0, 300)])
def test_chunk_full_size_workloads_sampled(idx, key_mode, n):
    """Chunk attention at the other workloads' full shapes (one layer of each
    distinct precision pair, batch cut to 2): Qwen2.5-7B-shaped with 7 query
    heads per kv head and per-token keys, KVmix's 800/384-token windows and
    its K3V4 orientation.  Sampled (unit, query) rows against fp64."""
    w = W.workload(idx)
    if key_mode:
        w = W.scaled(w, layers=tuple((kb, vb, r, key_mode, rpc) for kb, vb, r, _, rpc in map(W.spec_fields, w.layers)))
    w = W.scaled(w, batch=2)
    seen, layers = set(), []
    for l, lay in enumerate(w.layers):
        if lay not in seen:
            seen.add(lay)
            layers.append(l)
    T, D, Hkv, Hq = w.context, w.head_dim, w.num_kv_heads, w.num_q_heads
    rep = Hq // Hkv
    gen = torch.Generator(device="cuda")
    gen.manual_seed(31)
    for l in layers[:3]:
        kb, vb, R, km, rpc = W.spec_fields(w.layers[l])
        cache = K.KVQCache([w.layers[l]], w.batch, Hq, Hkv, D, w.group_size, T)
        k, v = W.gen_kv(w, l, 0, T, device="cuda")
        cache.append(0, k, v)
        q = torch.randn((w.batch, Hq, n, D), generator=gen, device="cuda").half()
        out = cache.chunk_attn(0, q)
        torch.cuda.synchronize()
        assert cache.device_error() == 0
        on, qn = out.cpu().numpy(), q.cpu().numpy()
        kn, vn = k.cpu().numpy(), v.cpu().numpy()
        U = w.batch * Hkv
        for u in sorted({0, U - 1}):
            b, h = divmod(u, Hkv)
            ora = O.OracleLayerCache(1, 1, D, w.group_size, kb, vb, R, km, rpc)
            ora.append(kn[b:b + 1, h:h + 1], vn[b:b + 1, h:h + 1])
            kh, vh = ora.dequantized(0)
            got, exp = [], []
            for j in (0, rep - 1):
                for i in (0, n // 3, n - 1):
                    pos = T - n + i
                    exp.append(O.attention_fp64(qn[b, h * rep + j, i].astype(np.float64), kh[: pos + 1], vh[: pos + 1]))
                    got.append(on[b, h * rep + j, i])
            assert_attn_close(np.stack(got), np.stack(exp), f"workload {idx} layer {l} unit {u}")
        cache.close()


def test_chunk_long_context_sampled():
    """Llama-2-70B-shaped unit at 32K context (8 query heads per kv head,
    G = R = 128): the largest workspace offsets and tile counts.  Sampled
    rows of a 256-query chunk against fp64 attention."""
    w = W.scaled(W.workload(5), batch=1, num_kv_heads=2, num_q_heads=16, decode_steps=1)
    T, D, Hkv, Hq, G = w.context, w.head_dim, w.num_kv_heads, w.num_q_heads, w.group_size
    rep = Hq // Hkv
    n = 256
    l = 0
    kb, vb, R = w.layers[l][:3]
    cache = K.KVQCache([w.layers[l]], 1, Hq, Hkv, D, G, T)
    k, v = W.gen_kv(w, l, 0, T, device="cuda")
    cache.append(0, k, v)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(41)
    q = torch.randn((1, Hq, n, D), generator=gen, device="cuda").half()
    out = cache.chunk_attn(0, q)
    torch.cuda.synchronize()
    assert cache.device_error() == 0
    on, qn, kn, vn = out.cpu().numpy(), q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy()
    for h in range(Hkv):
        ora = O.OracleLayerCache(1, 1, D, G, kb, vb, R)
        ora.append(kn[:, h:h + 1], vn[:, h:h + 1])
        kh, vh = ora.dequantized(0)
        got, exp = [], []
        for j in (0, rep - 1):
            for i in (0, 100, n - 1):
                pos = T - n + i
                exp.append(O.attention_fp64(qn[0, h * rep + j, i].astype(np.float64), kh[: pos + 1], vh[: pos + 1]))
                got.append(on[0, h * rep + j, i])
        assert_attn_close(np.stack(got), np.stack(exp), f"32K kv head {h}")
    cache.close()
