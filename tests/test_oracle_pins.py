"""Pins for the oracle: values printed on the pages, hand-worked examples, closed
forms, invariants and brute force.  CPU only."""

import math
import os

import numpy as np
import pytest

from oracle import kvq_oracle as O


def _lines(path):
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# ---------------------------------------------------------------- formulas

def test_kv_bytes_examples(golden_dir):
    n = 0
    for line in _lines(os.path.join(golden_dir, "kv_bytes_examples.txt")):
        f = line.split()
        L, H, d, S, b, expect = (int(x) for x in f[:6])
        assert O.kv_cache_bytes(L, H, d, S, b) == expect
        n += 1
    assert n == 6


def test_kv_bytes_page_roundings():
    # "~10.7 GB", "~43 GB", "~8.59 GB" (decimal GB), "> 50 GB"
    assert round(O.kv_cache_bytes(80, 8, 128, 32768, 2) / 1e9, 1) == 10.7
    assert round(O.kv_cache_bytes(80, 8, 128, 131072, 2) / 1e9) == 43
    assert round(O.kv_cache_bytes(64, 4, 128, 65536, 2) / 1e9, 2) == 8.59
    assert O.kv_cache_bytes(80, 64, 128, 20000, 2) > 50e9
    # exercise 1's "2-bit ~2.15 GB (4x saving)" is the FP16 figure divided by 4,
    # as printed; the pure 2-bit code payload is FP16/8.
    fp16 = O.kv_cache_bytes(64, 4, 128, 65536, 2)
    assert round(fp16 / 4 / 1e9, 2) == 2.15
    assert O.kv_cache_bytes(64, 4, 128, 65536, 2 / 8) == fp16 / 8


def test_equivalent_bits(golden_dir):
    for line in _lines(os.path.join(golden_dir, "equivalent_bits.txt")):
        pairs_s, expect = line.split()
        pairs = [tuple(int(t) for t in p.split(":")) for p in pairs_s.split(",")]
        assert O.equivalent_bits(pairs) == pytest.approx(float(expect), abs=1e-12)
    # KVmix averages: keys 70/32 ~ 2.19, values 76/32 ~ 2.38
    k_avg = (6 * 3 + 26 * 2) / 32
    v_avg = (6 * 4 + 26 * 2) / 32
    assert round(k_avg, 2) == 2.19 and round(v_avg, 2) == 2.38
    # search-space sizes quoted by KVTuner section A2: 9^32 ~ 3.4e30, 5^6 = 15625
    assert f"{9 ** 32:.1e}" == "3.4e+30"
    assert 5 ** 6 == 15625


def test_equivalent_bits_workloads():
    from mixed_precision_quantized_quant_gb300 import workloads as W
    eq = [O.equivalent_bits([tuple(p[:2]) for p in W.workload(i).layers]) for i in range(1, 6)]
    assert eq[0] == 3.0
    assert eq[1] == 111 / 32 and round(eq[1], 2) == 3.47
    assert eq[2] == 4.0
    assert eq[3] == 2.28125
    assert eq[4] == 3.1875
    w3 = W.workload(3)
    assert w3.layers[0][:2] == (8, 8) and w3.layers[-1][:2] == (8, 8)
    assert set(p[:2] for p in w3.layers) <= {(8, 8), (8, 4), (4, 4), (4, 2)}
    w4 = W.workload(4)
    hi = [l for l, p in enumerate(w4.layers) if p[:2] == (4, 3)]
    assert len(hi) == 6
    assert all(p[2] == 800 for p in w4.layers if p[:2] == (4, 3))
    assert all(p[2] == 384 for p in w4.layers if p[:2] == (2, 2))
    # KVmix's own orientation (page: key 2.19 and value 2.38 average bits): K3V4 on 6 of 32 layers
    w6 = W.workload(6)
    kavg = sum(p[0] for p in w6.layers) / len(w6.layers)
    vavg = sum(p[1] for p in w6.layers) / len(w6.layers)
    assert (kavg, vavg) == (2.1875, 2.375) and (round(kavg, 2), round(vavg, 2)) == (2.19, 2.38)
    assert sorted(set(p[:2] for p in w6.layers)) == [(2, 2), (3, 4)]


# ---------------------------------------------------------------- quantizer

def _parse_q(line):
    bits, xs, codes, s, z = (p.strip() for p in line.split("|"))
    return (int(bits), np.array([float(t) for t in xs.split()], dtype=np.float16),
            np.array([int(t) for t in codes.split()]), float(s), float(z))


def test_quantizer_worked_examples(golden_dir):
    n = 0
    for line in _lines(os.path.join(golden_dir, "quantizer_worked.txt")):
        bits, x, codes, s, z = _parse_q(line)
        c, s16, z16 = O.quantize_values_tokens(x[None, :], bits)
        assert list(c[0]) == list(codes), line
        assert float(s16[0]) == s and float(z16[0]) == z
        # same numbers through the per-channel key path (a column)
        ck, sk, zk = O.quantize_keys_group(x[:, None], bits)
        assert list(ck[:, 0]) == list(codes)
        assert float(sk[0]) == s and float(zk[0]) == z
        n += 1
    assert n == 5


def test_quantizer_inexact_fp16_scale_worked(golden_dir):
    # the fp32 scale is not an fp16 value: the codes follow the stored fp16 scale,
    # and on these inputs they differ from codes taken with the fp32 scale
    n = 0
    for line in _lines(os.path.join(golden_dir, "quantizer_fp16_scale_worked.txt")):
        parts = [p.strip() for p in line.split("|")]
        bits, x, codes, s, z = _parse_q("|".join(parts[:5]))
        codes32 = [int(t) for t in parts[5].split()]
        c, s16, z16 = O.quantize_values_tokens(x[None, :], bits)
        assert list(c[0]) == list(codes), line
        assert float(s16[0]) == s and float(z16[0]) == z
        ck, sk, zk = O.quantize_keys_group(x[:, None], bits)
        assert list(ck[:, 0]) == list(codes)
        assert float(sk[0]) == s and float(zk[0]) == z
        assert list(codes) != codes32  # the fixture separates the two readings
        n += 1
    assert n == 2


def _parse_rows(field):
    return np.array([[float(t) for t in r.split()] for r in field.split(";")], dtype=np.float64)


def test_rel_error_worked(golden_dir):
    from fractions import Fraction
    n = 0
    for line in _lines(os.path.join(golden_dir, "rel_error_worked.txt")):
        xs, xh, frac = (p.strip() for p in line.split("|"))
        x, x_hat = _parse_rows(xs), _parse_rows(xh)
        assert O.rel_error(x, x_hat) == pytest.approx(float(Fraction(frac)), rel=1e-12, abs=0.0), line
        n += 1
    assert n == 2


def test_key_group_worked(golden_dir):
    lines = list(_lines(os.path.join(golden_dir, "key_group_worked.txt")))
    bits = int(lines[0].split()[1])
    i_tok = lines.index("tokens")
    i_cod = lines.index("codes")
    toks = np.array([[float(t) for t in l.split()] for l in lines[i_tok + 1:i_cod]], dtype=np.float16)
    codes = np.array([[int(t) for t in l.split()] for l in lines[i_cod + 1:i_cod + 1 + toks.shape[0]]])
    scale = [float(t) for t in lines[-2].split()[1:]]
    zero = [float(t) for t in lines[-1].split()[1:]]
    c, s, z = O.quantize_keys_group(toks, bits)
    assert (c == codes).all()
    assert [float(v) for v in s] == scale
    assert [float(v) for v in z] == zero


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_quantizer_error_bound_and_endpoints(bits):
    rng = np.random.default_rng(7 + bits)
    x = (rng.standard_normal((64, 128)) * rng.lognormal(0, 1, (64, 1)) + rng.normal(0, 3, (64, 1)))
    x = x.astype(np.float16)
    codes, s16, z16 = O.quantize_values_tokens(x, bits)
    xh = O.dequant_values(codes, s16, z16, bits)
    s = s16.astype(np.float64)[:, None] * np.ones((1, 128))
    qmax = np.full((1, 128), 2 ** bits - 1, dtype=np.float64)
    if bits == 3:
        two = O.is_slot10(128)[None, :]
        s = np.where(two, O.slot10_scale(s16).astype(np.float64)[:, None], s)
        qmax = np.where(two, 3.0, 7.0)
    err = np.abs(x.astype(np.float64) - xh)
    bound = s / 2 + 4 * 2.0 ** -24 * (np.abs(z16.astype(np.float64))[:, None] + qmax * s)
    assert (err <= bound).all()
    # min -> code 0, max -> code qmax
    mn_idx = x.astype(np.float64).argmin(axis=1)
    mx_idx = x.astype(np.float64).argmax(axis=1)
    rows = np.arange(64)
    assert (codes[rows, mn_idx] == 0).all()
    top = np.where(O.is_slot10(128)[mx_idx], 3, 2 ** bits - 1) if bits == 3 else 2 ** bits - 1
    assert (codes[rows, mx_idx] == top).all()


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quantizer_power_of_two_grid_exact(bits):
    # x = mn + k * delta with delta a power of two and the full range used:
    # s = delta exactly, codes = k, reconstruction exact.
    rng = np.random.default_rng(bits)
    delta = 2.0 ** -3
    mn = -1.25
    k = rng.integers(0, 2 ** bits, size=200)
    k[0], k[1] = 0, 2 ** bits - 1
    x = (mn + k * delta).astype(np.float16)
    c, s, z = O.quantize_keys_group(x[:, None], bits)
    assert float(s[0]) == delta and float(z[0]) == mn
    assert (c[:, 0] == k).all()
    assert (O.dequant_keys(c, s, z, bits)[:, 0] == x.astype(np.float64)).all()


def test_quantizer_constant_group_exact():
    x = np.full((32, 128), 1.5, dtype=np.float16)
    for bits in (2, 3, 4, 8):
        c, s, z = O.quantize_keys_group(x, bits)
        assert (c == 0).all() and (s == 0).all()
        assert (O.dequant_keys(c, s, z, bits) == 1.5).all()


def test_ties_half_to_even():
    # b = 2, min 0, max 3 -> s = 1; x = 0.5, 1.5, 2.5 -> 0, 2, 2
    x = np.array([0, 3, 0.5, 1.5, 2.5], dtype=np.float16)
    c, s, _ = O.quantize_values_tokens(x[None, :], 2)
    assert float(s[0]) == 1.0
    assert list(c[0, 2:]) == [0, 2, 2]


def test_three_bit_slot10_scale():
    # the 2-bit field of a 3-bit word uses s2 = (s*7)/3 over the same range:
    # with min 0 and max 7 (s = 1), s2 = 7/3 and codes of 0, 7/3, 14/3, 7 are 0..3
    d = 11
    v = np.zeros((1, d), dtype=np.float16)
    v[0, 0] = 7
    for val, code in ((0.0, 0), (2.33, 1), (4.66, 2), (7.0, 3), (1.2, 1), (1.1, 0)):
        v[0, 10] = val
        c, s, z = O.quantize_values_tokens(v, 3)
        assert float(s[0]) == 1.0
        assert c[0, 10] == code, (val, c[0, 10])


# ---------------------------------------------------------------- packing

def test_packing_worked(golden_dir):
    n = 0
    for line in _lines(os.path.join(golden_dir, "packing_worked.txt")):
        bits, codes, words = (p.strip() for p in line.split("|"))
        bits = int(bits)
        codes = np.array([[int(t) for t in codes.split()]], dtype=np.uint8)
        expect = [int(t, 16) for t in words.split()]
        got = O.pack_rows(codes, bits)
        assert [int(w) for w in got[0]] == expect, line
        assert (O.unpack_rows(got, bits, codes.shape[1]) == codes).all()
        n += 1
    assert n == 5


@pytest.mark.parametrize("bits,d", [(2, 64), (2, 128), (3, 64), (3, 128), (4, 64), (4, 128), (8, 64), (8, 128)])
def test_pack_roundtrip_random(bits, d):
    rng = np.random.default_rng(bits * 1000 + d)
    codes = rng.integers(0, 2 ** bits, size=(50, d)).astype(np.uint8)
    if bits == 3:
        codes[:, O.is_slot10(d)] &= 3
    w = O.pack_rows(codes, bits)
    assert w.shape == (50, O.words_per_row(d, bits))
    assert (O.unpack_rows(w, bits, d) == codes).all()
    # independent bit-level check: rebuild each word from a Python int
    for r in range(3):
        for wi in range(w.shape[1]):
            acc = 0
            if bits == 3:
                for j in range(11):
                    c = wi * 11 + j
                    if c < d:
                        acc |= int(codes[r, c]) << (30 if j == 10 else 3 * j)
            else:
                per = 32 // bits
                for j in range(per):
                    acc |= int(codes[r, wi * per + j]) << (bits * j)
            assert acc == int(w[r, wi])


def test_three_bit_density():
    # 11 codes per word: 12 words per 128-vector, against 13 for 10 per word;
    # channels 10, 21, ..., 120 sit in the 2-bit fields
    assert O.words_per_row(128, 3) == 12
    assert math.ceil(128 / 10) == 13
    assert list(np.nonzero(O.is_slot10(128))[0]) == list(range(10, 128, 11))


# ---------------------------------------------------------------- attention

def test_attention_closed_form():
    # d = 2; scores q.k/sqrt(2): 0 and ln 3 -> weights 1/4, 3/4
    q = np.array([1.0, 0.0])
    k = np.array([[0.0, 0.0], [math.log(3) * math.sqrt(2), 5.0]])
    v = np.array([[4.0, 0.0], [0.0, 8.0]])
    o = O.attention_fp64(q, k, v)
    assert np.allclose(o, [1.0, 6.0], atol=1e-14)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(3)
    for T in range(1, 9):
        d = 4
        q = rng.standard_normal(d)
        k = rng.standard_normal((T, d))
        v = rng.standard_normal((T, d))
        # hand-expanded: weights exp(s_t) / sum exp(s_j), no max subtraction
        s = [sum(q[c] * k[t, c] for c in range(d)) / 2.0 for t in range(T)]
        e = [math.exp(x) for x in s]
        tot = sum(e)
        expect = [sum(e[t] / tot * v[t, c] for t in range(T)) for c in range(d)]
        assert np.allclose(O.attention_fp64(q, k, v), expect, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    d = 16
    q = rng.standard_normal(d)
    v = rng.standard_normal((5, d))
    k = np.tile(rng.standard_normal(d), (5, 1))
    assert np.allclose(O.attention_fp64(q, k, v), v.mean(axis=0))
    assert np.allclose(O.attention_fp64(q, k[:1], v[:1]), v[0])


def test_gqa_head_mapping():
    # query head h reads kv head h // (Hq/Hkv): with constant keys the output
    # of every query head is the mean of its kv head's values
    Hq, Hkv, T, d = 8, 2, 6, 4
    rng = np.random.default_rng(5)
    q = rng.standard_normal((Hq, d))
    k = np.zeros((Hkv, T, d))
    v = rng.standard_normal((Hkv, T, d))
    out = O.gqa_attention_fp64(q, k, v)
    for h in range(Hq):
        assert np.allclose(out[h], v[h // 4].mean(axis=0))


def test_lemma1_dominant_key():
    # KVTuner appendix Lemma 1: with one dominant key, quantization does not
    # move the attention output: both outputs ~ v_i
    rng = np.random.default_rng(6)
    d, T = 128, 64
    q = rng.standard_normal(d).astype(np.float16).astype(np.float64)
    k = rng.standard_normal((T, d)) * 0.1
    i = 17
    k[i] = q / np.linalg.norm(q) * 60 * math.sqrt(d) / np.linalg.norm(q)
    k16 = k.astype(np.float16)
    v16 = rng.standard_normal((T, d)).astype(np.float16)
    sc = (k16.astype(np.float64) @ q) / math.sqrt(d)
    assert sc[i] - np.delete(sc, i).max() >= 30
    codes, s, z = O.quantize_keys_group(k16, 2)
    kh = O.dequant_keys(codes, s, z, 2)
    vc, vs, vz = O.quantize_values_tokens(v16, 2)
    vh = O.dequant_values(vc, vs, vz, 2)
    o_exact = O.attention_fp64(q, k16, vh)
    o_quant = O.attention_fp64(q, kh, vh)
    assert np.allclose(o_exact, vh[i], atol=1e-9)
    assert np.allclose(o_quant, vh[i], atol=1e-9)


# ---------------------------------------------------------------- error orderings

def test_drift_exercise_per_token_beats_per_channel():
    # KIVI notes exercise 4: V drifts (first half N(0,1), second half N(10,1));
    # per-channel 2-bit scales taken from the first half (clamped) against
    # per-token scales
    rng = np.random.default_rng(11)
    T, d, b = 1024, 128, 2
    v = np.concatenate([rng.standard_normal((T // 2, d)), rng.standard_normal((T // 2, d)) + 10])
    v = v.astype(np.float16)
    first = v[: T // 2]
    mn = first.min(axis=0)
    s = O.asym_scale(mn, first.max(axis=0), b)
    pc_codes = O.asym_codes(v, mn[None, :], s.astype(np.float32)[None, :], 2 ** b - 1)
    pc = pc_codes * s.astype(np.float64)[None, :] + mn.astype(np.float64)[None, :]
    tc, ts, tz = O.quantize_values_tokens(v, b)
    pt = O.dequant_values(tc, ts, tz, b)
    err_pc = np.abs(v.astype(np.float64) - pc).sum()
    err_pt = np.abs(v.astype(np.float64) - pt).sum()
    # expected: the stale grid clamps the second half near the first half's
    # per-channel max (~3), ~7 per element on half the tokens; per token the
    # 2-bit grid over N(.,1) (range ~5, s ~1.7) errs ~s/4 per element:
    # ratio ~ (0.5*7 + 0.5*0.5) / 0.43 ~ 8.7
    assert 6 < err_pc / err_pt < 12
    assert err_pt / v.size < 0.5


def test_table9_ordering_keys_per_channel_beat_per_token():
    # KVTuner appendix (Table 9): at 2 bits, per-channel key error e_k is lower
    # than per-token e_k when keys carry channel outliers
    from mixed_precision_quantized_quant_gb300 import workloads as W
    w = W.scaled(W.workload(2), batch=1, num_layers=1)
    k, _ = W.gen_kv(w, 0, 0, 256)
    k = k[0, 0].numpy()
    ek_pc = []
    for g in range(0, 256, 32):
        c, s, z = O.quantize_keys_group(k[g:g + 32], 2)
        ek_pc.append(O.dequant_keys(c, s, z, 2))
    kh_pc = np.concatenate(ek_pc)
    kh_pt = O.quantize_keys_per_token(k, 2)
    assert O.rel_error(k, kh_pc) < O.rel_error(k, kh_pt)


# ---------------------------------------------------------------- streaming state

def test_flush_state_examples():
    # R = G: a 4096-token prefill leaves every token quantized
    assert O.flush_state(4096, 32, 32) == (4096, 0)
    assert O.flush_state(4096 + 31, 32, 32) == (4096, 31)
    assert O.flush_state(4096 + 32, 32, 32) == (4128, 0)
    # per-layer windows of 800 and 384 tokens (G = 32)
    assert O.flush_state(4096, 800, 32) == (3328, 768)
    assert O.flush_state(4096, 384, 32) == (3744, 352)
    assert O.flush_state(0, 64, 64) == (0, 0)


def test_oracle_cache_streaming_matches_bulk():
    # appending in pieces or in one call gives the same records and ring
    rng = np.random.default_rng(12)
    B, H, d, G, R = 1, 2, 64, 32, 96
    k = rng.standard_normal((B, H, 300, d)).astype(np.float16)
    v = rng.standard_normal((B, H, 300, d)).astype(np.float16)
    a = O.OracleLayerCache(B, H, d, G, 4, 2, R)
    a.append(k, v)
    b = O.OracleLayerCache(B, H, d, G, 4, 2, R)
    pos = 0
    for n in (1, 7, 50, 33, 1, 1, 100, 107):
        b.append(k[:, :, pos:pos + n], v[:, :, pos:pos + n])
        pos += n
    assert pos == 300
    assert (a.n_q, a.r) == (b.n_q, b.r) == O.flush_state(300, R, G)
    for u in range(B * H):
        assert a.unit_records(u) == b.unit_records(u)
        ka, va = a.residual_ring(u)
        kb_, vb_ = b.residual_ring(u)
        assert (ka == kb_).all() and (va == vb_).all()
    # dequantized tokens: quantized groups are close, the residual is exact
    kh, vh = a.dequantized(0)
    assert kh.shape == (300, d)
    assert (kh[a.n_q:] == k[0, 0, a.n_q:].astype(np.float64)).all()
    assert np.abs(kh[: a.n_q] - k[0, 0, : a.n_q]).max() < 1.0


def test_record_layout_sizes():
    lay = O.record_layout(128, 32, 4, 2)
    assert lay["wk"] == 16 and lay["wv"] == 8
    assert lay["bytes"] == 32 * 64 + 32 * 32 + 4 * 128 + 4 * 32
    lay3 = O.record_layout(128, 32, 4, 3)
    assert lay3["wv"] == 12
    for d in (64, 128):
        for G in (32, 64, 128):
            for kb in O.BITS_ALLOWED:
                for vb in O.BITS_ALLOWED:
                    assert O.record_layout(d, G, kb, vb)["bytes"] % 16 == 0


@pytest.mark.parametrize("d", [64, 128])
def test_key_scale_rows_stored_chunk_order_worked(d):
    # Per-channel key scale and zero rows are stored in 8-channel chunks, chunk j
    # of each channel quarter side by side.  Worked orders (natural chunk index
    # at each stored position), written out by hand:
    #   d = 64:  quarters {0,1} {2,3} {4,5} {6,7} -> 0 2 4 6 | 1 3 5 7
    #   d = 128: quarters {0..3} {4..7} {8..11} {12..15}
    #            -> 0 4 8 12 | 1 5 9 13 | 2 6 10 14 | 3 7 11 15
    hand = {64: [0, 2, 4, 6, 1, 3, 5, 7],
            128: [0, 4, 8, 12, 1, 5, 9, 13, 2, 6, 10, 14, 3, 7, 11, 15]}[d]
    assert list(O.key_scale_chunk_order(d)) == hand
    # a group whose channel c spans [c, c + 1]: zero row = c, scale row = 1/qmax
    G, bits = 32, 4
    k = (np.arange(d)[None, :] + (np.arange(G)[:, None] % 2)).astype(np.float16)
    v = np.zeros((G, d), dtype=np.float16)
    rec = O.build_group_record(k, v, bits, 2)
    lay = O.record_layout(d, G, bits, 2)
    buf = np.frombuffer(rec, dtype=np.uint8)
    zero_row = buf[lay["k_zero"]:lay["v_scale"]].view(np.float16).astype(np.int64)
    expect = np.concatenate([np.arange(8 * c, 8 * c + 8) for c in hand])
    assert (zero_row == expect).all()
    scale_row = buf[lay["k_scale"]:lay["k_zero"]].view(np.float16)
    assert (scale_row == np.float16(1.0 / 15.0)).all()
    # and the parse restores every channel: dequantized keys are exact here
    kh, _ = O.parse_group_record(rec, d, G, bits, 2)
    assert np.abs(kh - k.astype(np.float64)).max() <= 2.0 ** -9
    # 3-bit keys keep the natural channel order
    rec3 = O.build_group_record(k, v, 3, 2)
    lay3 = O.record_layout(d, G, 3, 2)
    buf3 = np.frombuffer(rec3, dtype=np.uint8)
    assert (buf3[lay3["k_zero"]:lay3["v_scale"]].view(np.float16).astype(np.int64) == np.arange(d)).all()


def test_code_row_word_order_worked():
    # Stored word order of code rows, written out by hand for rows whose packed
    # words are 0, 1, 2, ... (entry i = the packed word kept at index i).
    a16, a32 = list(range(16)), list(range(32))
    swap4 = [4, 5, 6, 7, 0, 1, 2, 3]
    k8_row1 = [w + 8 * b for b in range(4) for w in swap4]            # 8-bit keys, d = 128, odd row
    v16_row2 = list(range(8, 16)) + list(range(8))                    # 16-word value rows, t & 2
    v32 = {1: list(range(8, 16)) + list(range(8)) + list(range(24, 32)) + list(range(16, 24)),
           2: list(range(16, 32)) + list(range(16)),
           3: list(range(24, 32)) + list(range(16, 24)) + list(range(8, 16)) + list(range(8))}
    rows32 = np.tile(np.arange(32, dtype=np.uint32), (4, 1))
    rows16 = np.tile(np.arange(16, dtype=np.uint32), (4, 1))
    k = O.code_rows_store(rows32, True)
    assert list(k[0]) == a32 and list(k[1]) == k8_row1 and list(k[2]) == a32 and list(k[3]) == k8_row1
    v = O.code_rows_store(rows16, False)
    assert list(v[0]) == a16 and list(v[1]) == a16 and list(v[2]) == v16_row2 and list(v[3]) == v16_row2
    v = O.code_rows_store(rows32, False)
    assert list(v[0]) == a32 and all(list(v[t]) == v32[t] for t in (1, 2, 3))
    # 16-word key rows (4-bit, d = 128) and 8-word rows are kept as packed
    assert (O.code_rows_store(rows16, True) == rows16).all()
    assert (O.code_rows_store(rows32[:, :8], False) == rows32[:, :8]).all()
    for is_key, rows in ((True, rows32), (False, rows16), (False, rows32)):
        assert (O.code_rows_load(O.code_rows_store(rows, is_key), is_key) == rows).all()
    # through a record: an 8-bit key code row and a 4-bit value code row in storage order
    G, d = 32, 128
    rng = np.random.default_rng(5)
    kx = rng.standard_normal((G, d)).astype(np.float16)
    vx = rng.standard_normal((G, d)).astype(np.float16)
    rec = O.build_group_record(kx, vx, 8, 4)
    lay = O.record_layout(d, G, 8, 4)
    buf = np.frombuffer(rec, dtype=np.uint8)
    kc, _, _ = O.quantize_keys_group(kx, 8)
    vc, _, _ = O.quantize_values_tokens(vx, 4)
    kst = buf[lay["k_codes"]:lay["v_codes"]].view(np.uint32).reshape(G, 32)
    vst = buf[lay["v_codes"]:lay["k_scale"]].view(np.uint32).reshape(G, 16)
    assert (kst[1] == O.pack_rows(kc, 8)[1][k8_row1]).all()
    assert (vst[2] == O.pack_rows(vc, 4)[2][v16_row2]).all()
    assert (vst[0] == O.pack_rows(vc, 4)[0]).all()


# ---------------------------------------------------------------------------
# Per-token-asym key mode ([KVTuner] A3-A4: the second quantization mode,
# keys quantized per token like values)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [2, 4, 8])
def test_per_token_key_record_quantizes_along_tokens(bits):
    # keys with strong channel outliers: per token, each token's min and max
    # must land on codes 0 and 2^b - 1 and every element stay within s_t/2
    rng = np.random.default_rng(100 + bits)
    G, d = 32, 128
    k = rng.standard_normal((G, d)) * 1.5
    k[:, 3] *= 12.0
    k = k.astype(np.float16)
    v = rng.standard_normal((G, d)).astype(np.float16)
    rec = O.build_group_record(k, v, bits, 4, O.KEY_PER_TOKEN)
    lay = O.record_layout(d, G, bits, 4, O.KEY_PER_TOKEN)
    assert len(rec) == lay["bytes"]
    buf = np.frombuffer(rec, dtype=np.uint8)
    codes = O.unpack_rows(O.code_rows_load(buf[lay["k_codes"]:lay["v_codes"]].view(np.uint32).reshape(G, lay["wk"]), True), bits, d)
    ksz = buf[lay["k_scale"]:lay["v_scale"]].view(np.float16).reshape(G, 2)
    kf = k.astype(np.float64)
    rows = np.arange(G)
    assert (codes[rows, kf.argmin(axis=1)] == 0).all()
    assert (codes[rows, kf.argmax(axis=1)] == 2 ** bits - 1).all()
    assert (ksz[:, 1] == k.min(axis=1)).all()                        # zero = per-token min
    s = ksz[:, 0].astype(np.float64)[:, None]
    kh, vh = O.parse_group_record(rec, d, G, bits, 4, O.KEY_PER_TOKEN)
    bound = s / 2 + 4 * 2.0 ** -24 * (np.abs(ksz[:, 1].astype(np.float64))[:, None] + (2 ** bits - 1) * s)
    assert (np.abs(kf - kh) <= bound).all()
    # values are unaffected by the key mode
    _, vh0 = O.parse_group_record(O.build_group_record(k, v, bits, 4), d, G, bits, 4)
    assert (vh == vh0).all()
    # with outlier channels, per-token keys lose far more than per-channel ones
    kh0, _ = O.parse_group_record(O.build_group_record(k, v, bits, 4), d, G, bits, 4)
    assert np.abs(kf - kh).mean() > np.abs(kf - kh0).mean()


def test_per_token_key_record_layout_sizes():
    for d in (64, 128):
        for G in (32, 64, 128):
            for kb in (2, 4, 8):
                for vb in O.BITS_ALLOWED:
                    lay = O.record_layout(d, G, kb, vb, O.KEY_PER_TOKEN)
                    assert lay["bytes"] == 4 * G * (lay["wk"] + lay["wv"]) + 4 * G + 4 * G
                    assert lay["bytes"] % 16 == 0


def test_per_token_key_cache_streaming_matches_bulk():
    rng = np.random.default_rng(13)
    B, H, d, G, R = 1, 2, 64, 32, 64
    k = rng.standard_normal((B, H, 200, d)).astype(np.float16)
    v = rng.standard_normal((B, H, 200, d)).astype(np.float16)
    a = O.OracleLayerCache(B, H, d, G, 8, 2, R, O.KEY_PER_TOKEN)
    a.append(k, v)
    b = O.OracleLayerCache(B, H, d, G, 8, 2, R, O.KEY_PER_TOKEN)
    pos = 0
    for n in (3, 61, 1, 1, 90, 44):
        b.append(k[:, :, pos:pos + n], v[:, :, pos:pos + n])
        pos += n
    assert (a.n_q, a.r) == (b.n_q, b.r) == O.flush_state(200, R, G)
    for u in range(B * H):
        assert a.unit_records(u) == b.unit_records(u)
    # attention over per-token-quantized 8-bit keys stays close to exact attention
    q = rng.standard_normal((B, H, d)).astype(np.float16)
    kh, vh = a.dequantized(0)
    o = O.attention_fp64(q[0, 0].astype(np.float64), kh, vh)
    oe = O.attention_fp64(q[0, 0].astype(np.float64), k[0, 0].astype(np.float64), vh)
    assert np.abs(o - oe).max() < 0.05


# ---------------------------------------------------------------------------
# Intra-layer pair pruning ([KVTuner] A2, two-stage search-space pruning, and
# Table 3 of its A3 observations)
# ---------------------------------------------------------------------------

def _pruning_case():
    from mixed_precision_quantized_quant_gb300 import workloads as W
    w = W.scaled(W.workload(2), batch=1, num_kv_heads=2, num_q_heads=8, context=512, decode_steps=4)
    k, v = W.gen_kv(w, 5, 0, w.context)
    qs = [W.gen_q(w, 5, s).numpy() for s in range(2)]
    return k.numpy(), v.numpy(), qs


def test_pareto_front_keeps_kvtuners_pairs():
    # On keys with channel outliers and values with drifting means, the e_o
    # front over {2, 4, 8}^2 is the five pairs KVTuner's pruning keeps:
    # KV2, K4V2, KV4, K8V4, KV8 (K2V4, K8V2, K2V8 and K4V8 are dominated).
    k, v, qs = _pruning_case()
    pairs = [(kb, vb) for kb in (2, 4, 8) for vb in (2, 4, 8)]
    err = O.pair_output_errors(k, v, qs, pairs, 32, 32)
    assert O.pareto_front(err) == [(2, 2), (4, 2), (4, 4), (8, 4), (8, 8)]
    # Table 3's reading: at the same memory, precise keys beat precise values
    assert err[(4, 2)] < err[(2, 4)] and err[(8, 4)] < err[(4, 8)]
    # more bits on both sides never hurts here
    assert err[(8, 8)] < err[(4, 4)] < err[(2, 2)]


def test_pareto_front_filter():
    err = {(8, 8): 0.001, (8, 4): 0.01, (4, 8): 0.02, (4, 4): 0.015, (4, 2): 0.05, (2, 4): 0.2, (2, 2): 0.3}
    # K4V8 (6 bits, 0.02) is dominated by K8V4 (6 bits, 0.01); K2V4 by K4V2
    assert O.pareto_front(err) == [(2, 2), (4, 2), (4, 4), (8, 4), (8, 8)]
    # fewer bits at an equal error dominates; a tie in both coordinates does not
    assert O.pareto_front({(4, 4): 0.1, (2, 8): 0.1}) == [(4, 4)]
    assert sorted(O.pareto_front({(8, 2): 0.1, (2, 8): 0.1})) == [(2, 8), (8, 2)]


# ---------------------------------------------------------------------------
# Chunk attention: causal queries over the cache ([KVTuner] A2 calibration,
# prefill over the dequantized cache; A3 attention)
# ---------------------------------------------------------------------------

def _sdpa_bottom_right(q, k, v):
    """torch's attention routine (fp64, CPU) with an explicit mask: query i of
    n sees keys 0 .. T - n + i.  q [Hq, n, d], k/v [Hq, T, d]."""
    import torch
    n, T = q.shape[1], k.shape[1]
    mask = torch.ones(n, T, dtype=torch.bool).tril(diagonal=T - n)
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=mask).numpy()


@pytest.mark.parametrize("kb,vb,km,T,n", [(4, 2, 0, 160, 160), (3, 3, 0, 150, 37), (8, 4, 1, 129, 64),
                                          (2, 8, 0, 96, 1)])
def test_chunk_attention_matches_library_routine(kb, vb, km, T, n):
    rng = np.random.default_rng(11)
    B, H, rep, d, G = 1, 2, 3, 64, 32
    k = (rng.standard_normal((B, H, T, d)) * (1 + 4 * (np.arange(d) % 9 == 0))).astype(np.float16)
    v = rng.standard_normal((B, H, T, d)).astype(np.float16)
    q = rng.standard_normal((B, H * rep, n, d)).astype(np.float16)
    c = O.OracleLayerCache(B, H, d, G, kb, vb, G, km)
    c.append(k[:, :, : T // 2], v[:, :, : T // 2])
    c.append(k[:, :, T // 2:], v[:, :, T // 2:])
    assert c.n_q > 0
    got = c.attend_chunk(q)
    for h in range(H):
        kh, vh = c.dequantized(h)
        exp = _sdpa_bottom_right(q[0, h * rep:(h + 1) * rep].astype(np.float64),
                                 np.broadcast_to(kh, (rep,) + kh.shape).copy(),
                                 np.broadcast_to(vh, (rep,) + vh.shape).copy())
        np.testing.assert_allclose(got[0, h * rep:(h + 1) * rep], exp, rtol=1e-12, atol=1e-12)


def test_chunk_attention_full_causal_prefill_without_quantization():
    # window longer than the prompt: nothing is quantized and n = T is the
    # plain causal prefill attention over the fp16 K and V
    import torch
    rng = np.random.default_rng(12)
    T, d = 70, 64
    k = rng.standard_normal((1, 1, T, d)).astype(np.float16)
    v = rng.standard_normal((1, 1, T, d)).astype(np.float16)
    q = rng.standard_normal((1, 2, T, d)).astype(np.float16)
    c = O.OracleLayerCache(1, 1, d, 32, 2, 2, 96)
    c.append(k, v)
    assert c.n_q == 0
    got = c.attend_chunk(q)
    exp = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64)), torch.from_numpy(np.repeat(k, 2, 1).astype(np.float64)),
        torch.from_numpy(np.repeat(v, 2, 1).astype(np.float64)), is_causal=True).numpy()
    np.testing.assert_allclose(got, exp, rtol=1e-12, atol=1e-12)


def test_chunk_attention_equal_keys_give_running_means():
    # all keys equal: every visible token has the same weight, so query i
    # returns the mean of the values at positions 0 .. T - n + i
    rng = np.random.default_rng(13)
    T, n, d = 200, 50, 64
    k = np.broadcast_to(rng.standard_normal(d).astype(np.float16), (1, 1, T, d)).copy()
    v = rng.standard_normal((1, 1, T, d)).astype(np.float16)
    q = rng.standard_normal((1, 1, n, d)).astype(np.float16)
    c = O.OracleLayerCache(1, 1, d, 32, 8, 8, 256)
    c.append(k, v)
    got = c.attend_chunk(q)[0, 0]
    run = np.cumsum(v[0, 0].astype(np.float64), axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(got, run[T - n:], rtol=1e-9, atol=1e-12)


def test_chunk_attention_rejects_bad_lengths():
    c = O.OracleLayerCache(1, 1, 64, 32, 4, 4, 32)
    c.append(np.zeros((1, 1, 5, 64), np.float16), np.zeros((1, 1, 5, 64), np.float16))
    with pytest.raises(ValueError):
        c.attend_chunk(np.zeros((1, 1, 6, 64), np.float16))


# ---------------------------------------------------------------- KVmix dynamic window

def test_rpc_window_worked(golden_dir):
    # token-by-token state of one unit against the hand-worked sequence; the
    # cache holds tiny rows (d = 64) since only the counts are checked
    rows = [tuple(int(t) for t in line.split("|")) for line in _lines(os.path.join(golden_dir, "rpc_window_worked.txt"))]
    assert len(rows) == 11
    for pct, R in sorted({(r[0], r[1]) for r in rows}):
        want = {r[2]: r[3:] for r in rows if r[:2] == (pct, R)}
        c = O.OracleLayerCache(1, 1, 64, 32, 2, 2, R, rpc_percent=pct)
        rng = np.random.default_rng(pct)
        c.append(rng.standard_normal((1, 1, 4096, 64)).astype(np.float16),
                 rng.standard_normal((1, 1, 4096, 64)).astype(np.float16))
        for step in range(max(want) + 1):
            if step:
                c.append(rng.standard_normal((1, 1, 1, 64)).astype(np.float16),
                         rng.standard_normal((1, 1, 1, 64)).astype(np.float16))
            if step in want:
                assert (c.n_q, c.r, c.bound) == want[step], (pct, step)
            assert c.r < c.bound and c.n_q + c.r == 4096 + step


def test_rpc_shrink_bound_closed_form():
    # G * max(1, floor(p * C / (100 G))): a multiple of G, at least G, at most C
    for G in (32, 64, 128):
        for p in (1, 10, 20, 50, 100):
            for C in range(G, 40 * G + 1, G):
                b = O.shrink_bound(C, p, G)
                assert b % G == 0 and G <= b <= C
                assert b == G * max(1, (p * C) // (100 * G))
    assert O.shrink_bound(800, 20, 32) == 160 and O.shrink_bound(384, 10, 32) == 32


def test_rpc_zero_is_the_static_window():
    # p = 0 keeps the bound at R: the same records and window as the plain cache
    rng = np.random.default_rng(3)
    a = O.OracleLayerCache(1, 2, 64, 32, 4, 2, 96)
    b = O.OracleLayerCache(1, 2, 64, 32, 4, 2, 96, rpc_percent=0)
    for n in [100, 1, 1, 40, 1] + [1] * 70:
        k = rng.standard_normal((1, 2, n, 64)).astype(np.float16)
        v = rng.standard_normal((1, 2, n, 64)).astype(np.float16)
        a.append(k, v)
        b.append(k, v)
        assert (a.n_q, a.r) == (b.n_q, b.r) == O.flush_state(a.total, 96, 32)
    assert a.records == b.records and b.bound == 96


def test_rpc_records_and_ring_after_a_shrink():
    # the groups quantized in one shrinking step are the oldest window tokens in
    # order, each a plain group record; the live window keeps ring slots i mod R
    rng = np.random.default_rng(5)
    G, R, d = 32, 160, 64
    c = O.OracleLayerCache(1, 1, d, G, 4, 2, R, rpc_percent=20)
    toks_k, toks_v = [], []
    def push(n):
        k = rng.standard_normal((1, 1, n, d)).astype(np.float16)
        v = rng.standard_normal((1, 1, n, d)).astype(np.float16)
        toks_k.append(k[0, 0]); toks_v.append(v[0, 0])
        c.append(k, v)
    push(300)                      # 300 - 32k < 160 at k = 5: quantized 160, window 140
    assert (c.n_q, c.r, c.bound) == (160, 140, 160)
    for _ in range(20):            # the 20th step brings the window to 160 -> bound 32, 5 groups
        push(1)
    assert (c.n_q, c.r, c.bound) == (320, 0, 32)
    allk, allv = np.concatenate(toks_k), np.concatenate(toks_v)
    for j, rec in enumerate(c.records[0]):
        assert rec == O.build_group_record(allk[j * G:(j + 1) * G], allv[j * G:(j + 1) * G], 4, 2)
    push(1)
    push(1)
    allk = np.concatenate(toks_k)
    rk, _ = c.residual_ring(0)
    assert (c.n_q, c.r) == (320, 2)
    assert (rk[320 % R] == allk[320]).all() and (rk[321 % R] == allk[321]).all()


# ---------------------------------------------------------------- decode attention of the cache model

def _sdpa_fp64(q, k, v):
    """torch's attention in fp64: q [Hq, d], k/v [T, d] shared by every head."""
    import torch
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[:, None, :]
    kt = torch.from_numpy(np.asarray(k, dtype=np.float64))[None].expand(qt.shape[0], -1, -1)
    vt = torch.from_numpy(np.asarray(v, dtype=np.float64))[None].expand(qt.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0].numpy()


@pytest.mark.parametrize("kb,vb,km", [(4, 2, 0), (3, 3, 0), (8, 4, 1), (2, 2, 0)])
def test_attend_exact_grid_equals_library_attention(kb, vb, km):
    # [KVTuner] A3 attention over the cache: with every key group and value
    # token on a grid its quantizer reconstructs exactly (min, max and the
    # values in between multiples of a power-of-two step), the dequantized
    # cache is the fp16 K and V themselves, so the cache model's decode
    # attention (append, then attend over groups and window) must equal
    # torch's fp64 attention over the raw K and V, head mapping included.
    rng = np.random.default_rng(21)
    B, H, rep, d, G, R, T = 2, 2, 3, 64, 32, 64, 150
    qk, qv = (1 << kb) - 1, (1 << vb) - 1
    # keys: per channel over each group (or per token) a grid of step 2^-2,
    # every channel of every group touching both ends of its code range
    codes_k = rng.integers(0, qk + 1, (B, H, T, d))
    codes_v = rng.integers(0, qv + 1, (B, H, T, d))
    if km == 0:
        for g0 in range(0, T, G):
            codes_k[:, :, g0, :] = 0
            codes_k[:, :, min(g0 + 1, T - 1), :] = qk
    else:
        codes_k[..., 0] = 0
        codes_k[..., 1] = qk
    codes_v[..., 0] = 0
    codes_v[..., 1] = qv
    # 3-bit words: the 2-bit field (channel 11j + 10) is scaled by s2 = 7s/3,
    # not a power of two, so it holds only its range's minimum here
    slot10 = (np.arange(d) % 11) == 10
    if kb == 3:
        codes_k[..., slot10] = 0
    if vb == 3:
        codes_v[..., slot10] = 0
    # per channel keys: a per-channel offset; per-token keys and values: a
    # per-token offset (the minimum of each quantized row or column)
    base_k = rng.integers(-8, 8, (B, H, 1, d) if km == 0 else (B, H, T, 1)) * 0.5
    base_v = rng.integers(-8, 8, (B, H, T, 1)) * 0.5
    k = (base_k + codes_k * 0.25).astype(np.float16)
    v = (base_v + codes_v * 0.25).astype(np.float16)
    q = rng.standard_normal((B, H * rep, d)).astype(np.float16)
    c = O.OracleLayerCache(B, H, d, G, kb, vb, R, km)
    c.append(k[:, :, :100], v[:, :, :100])
    c.append(k[:, :, 100:], v[:, :, 100:])
    assert c.n_q > 0 and c.r > 0
    got = c.attend(q)
    for b in range(B):
        for h in range(H):
            exp = _sdpa_fp64(q[b, h * rep:(h + 1) * rep], k[b, h], v[b, h])
            np.testing.assert_allclose(got[b, h * rep:(h + 1) * rep], exp, rtol=1e-12, atol=1e-12)


def test_attend_window_only_equals_library_attention():
    # a window longer than the context: nothing is quantized and the decode
    # attention is plain fp64 attention over the fp16 K and V
    rng = np.random.default_rng(22)
    B, H, rep, d, G = 1, 2, 4, 128, 32
    k = rng.standard_normal((B, H, 90, d)).astype(np.float16)
    v = rng.standard_normal((B, H, 90, d)).astype(np.float16)
    q = rng.standard_normal((B, H * rep, d)).astype(np.float16)
    c = O.OracleLayerCache(B, H, d, G, 4, 2, 128)
    c.append(k, v)
    assert c.n_q == 0
    got = c.attend(q)
    for h in range(H):
        np.testing.assert_allclose(got[0, h * rep:(h + 1) * rep], _sdpa_fp64(q[0, h * rep:(h + 1) * rep], k[0, h], v[0, h]),
                                   rtol=1e-12, atol=1e-12)


def test_live_ring_slots_worked():
    # flush rule with R = 64, G = 32 ([KIVI notes] 6.2): after 100 tokens two
    # groups (64 tokens) are quantized and tokens 64..99 sit in slots 0..35;
    # after 70 tokens one group is quantized and tokens 32..69 sit in slots
    # 32..63 then 0..5
    d = 64
    for T, nq, slots in ((100, 64, list(range(36))), (70, 32, list(range(32, 64)) + list(range(6)))):
        c = O.OracleLayerCache(1, 1, d, 32, 4, 2, 64)
        x = np.zeros((1, 1, T, d), dtype=np.float16)
        c.append(x, x)
        assert c.n_q == nq
        assert c.live_ring_slots().tolist() == slots
