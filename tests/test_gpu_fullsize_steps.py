"""Full-size parity over every decode step, in the benchmark's launch
configuration (the captured decode step: appends on a forked stream, each
layer's decode a programmatic dependent of the previous one).

* Llama-3.1-8B- and Qwen2.5-7B-shaped workloads: every layer, two (batch, kv
  head) units per layer, attention checked at every decode step, group
  records and the FP16 window compared byte for byte at every step that
  flushes a key group and at the last one;
* KVmix-shaped workloads (shrinking RPC windows, both orientations): one
  layer and one unit per precision pair, every one of the 256 decode steps.

The oracle's dequantization of a unit's groups is kept between steps here
(a group record never changes once written), and attention is the oracle's
fp64 attention over those values and the unit's FP16 tokens."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import kvq_oracle as O
from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import workloads as W
from tests.kvq_testutil import assert_attn_close, gpu_unit_records, gpu_unit_ring

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    K.load()


class _Tracked:
    """One unit's oracle cache with its dequantized groups kept up to date."""

    def __init__(self, w, spec):
        kb, vb, R, km, rpc = W.spec_fields(spec)
        self.ora = O.OracleLayerCache(1, 1, w.head_dim, w.group_size, kb, vb, R, km, rpc)
        self.kb, self.vb, self.km = kb, vb, km
        self.ngroups = 0
        self.kq = np.zeros((0, w.head_dim))
        self.vq = np.zeros((0, w.head_dim))

    def append(self, k, v):
        self.ora.append(k, v)
        o = self.ora
        new_k, new_v = [self.kq], [self.vq]
        while self.ngroups < len(o.records[0]):
            kh, vh = O.parse_group_record(o.records[0][self.ngroups], o.d, o.G, self.kb, self.vb, self.km)
            new_k.append(kh)
            new_v.append(vh)
            self.ngroups += 1
        if len(new_k) > 1:
            self.kq = np.concatenate(new_k, axis=0)
            self.vq = np.concatenate(new_v, axis=0)

    def attend(self, q_heads):
        o = self.ora
        kk = np.concatenate([self.kq, o.pend_k[0].astype(np.float64)], axis=0)
        vv = np.concatenate([self.vq, o.pend_v[0].astype(np.float64)], axis=0)
        return np.stack([O.attention_fp64(qh.astype(np.float64), kk, vv) for qh in q_heads])


def _check_bytes(cache, layer, u, tr):
    assert gpu_unit_records(cache, layer, u) == tr.ora.unit_records(0), f"records layer {layer} unit {u}"
    live = tr.ora.live_ring_slots()
    if len(live):
        gk, gv = gpu_unit_ring(cache, layer, u)
        ok_, ov_ = tr.ora.residual_ring(0)
        assert np.array_equal(gk[live].view(np.uint16), ok_[live].view(np.uint16)), f"ring K layer {layer} unit {u}"
        assert np.array_equal(gv[live].view(np.uint16), ov_[live].view(np.uint16)), f"ring V layer {layer} unit {u}"


def _unit(x, u, H):
    b, h = divmod(u, H)
    return x[b:b + 1, h:h + 1].cpu().numpy()


def _run(w, layers, units_of, steps):
    """Prefill the listed layers of w, then `steps` captured decode steps;
    units_of(i) lists the units checked on the i-th listed layer."""
    L = len(layers)
    sub = [w.layers[l] for l in layers]
    U = w.batch * w.num_kv_heads
    rep = w.num_q_heads // w.num_kv_heads
    cache = K.KVQCache(sub, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size, w.context + steps)
    tracked = {}
    for i, l in enumerate(layers):
        k, v = W.gen_kv(w, l, 0, w.context, device="cuda")
        cache.append(i, k, v)
        for u in units_of(i):
            assert 0 <= u < U
            t = _Tracked(w, w.layers[l])
            t.append(_unit(k, u, w.num_kv_heads), _unit(v, u, w.num_kv_heads))
            tracked[(i, u)] = t
        del k, v
    for (i, u), t in tracked.items():
        _check_bytes(cache, i, u, t)
    stream = torch.cuda.Stream()
    kc = torch.empty((L, w.batch, w.num_kv_heads, 1, w.head_dim), dtype=torch.float16, device="cuda")
    vc = torch.empty_like(kc)
    qc = torch.empty((L, w.batch, w.num_q_heads, w.head_dim), dtype=torch.float16, device="cuda")
    out = torch.empty((L, w.batch, w.num_q_heads, w.head_dim), device="cuda")
    for s in range(steps):
        for i, l in enumerate(layers):
            k1, v1 = W.gen_kv(w, l, w.context + s, 1, device="cuda")
            kc[i].copy_(k1)
            vc[i].copy_(v1)
            qc[i].copy_(W.gen_q(w, l, s, device="cuda"))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            cache.decode_step([kc[i] for i in range(L)], [vc[i] for i in range(L)], [qc[i] for i in range(L)],
                              [out[i] for i in range(L)], stream=stream)
        stream.synchronize()
        outn, qn = out.cpu().numpy(), qc.cpu().numpy()
        kn, vn = kc.cpu().numpy(), vc.cpu().numpy()
        for (i, u), t in tracked.items():
            b, h = divmod(u, w.num_kv_heads)
            nq0 = t.ora.n_q
            t.append(kn[i, b:b + 1, h:h + 1], vn[i, b:b + 1, h:h + 1])
            if t.ora.n_q != nq0 or s == steps - 1:
                _check_bytes(cache, i, u, t)
            exp = t.attend(qn[i, b, h * rep:(h + 1) * rep])
            assert_attn_close(outn[i, b, h * rep:(h + 1) * rep], exp, f"{w.name} layer {layers[i]} step {s} unit {u}")
    assert cache.device_error() == 0
    cache.close()


@pytest.mark.parametrize("idx", [2, 3])
def test_every_step_every_layer_two_units(idx):
    w = W.workload(idx)
    U = w.batch * w.num_kv_heads
    layers = list(range(w.num_layers))
    _run(w, layers, lambda i: sorted({(7 * i + 1) % U, U - 1 - (3 * i) % U}), w.decode_steps)


@pytest.mark.parametrize("idx", [4, 6])
def test_kvmix_all_steps_one_unit_per_pair(idx):
    w = W.workload(idx)
    U = w.batch * w.num_kv_heads
    first = {}
    for l, spec in enumerate(w.layers):
        first.setdefault(W.spec_fields(spec)[:2], l)
    layers = sorted(first.values())
    _run(w, layers, lambda i: [(97 * layers[i] + 13) % U], w.decode_steps)
