"""State snapshots (kvq_state_save / kvq_state_restore): a restored cache
replays a window of decode steps bit for bit, through the step graph and
through per-layer calls with multi-token appends; a snapshot whose counters
describe no reachable state is refused before anything changes."""

import pytest
import torch

from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# a static window, a shrinking (RPC) window, per-token keys and a 3-bit pair
LAYERS = ((8, 4, 64), (2, 2, 128, 0, 20), (4, 2, 64, 1), (4, 3, 64, 0, 50))


def _workload():
    return W.scaled(W.workload(2), batch=2, num_layers=len(LAYERS), context=300, decode_steps=140, layers=LAYERS)


def _prefilled(w):
    c = K.KVQCache(w.layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size, w.total_tokens)
    for l in range(w.num_layers):
        k, v = W.gen_kv(w, l, 0, w.context, device="cuda")
        c.append(l, k, v)
    return c


def _views(c, L):
    return [{k: v for k, v in c.view(l).items() if k in ("tokens", "quantized_tokens", "window_bound")}
            for l in range(L)]


def test_restore_replays_step_graph_bit_exact():
    w = _workload()
    L = w.num_layers
    c = _prefilled(w)
    stream = torch.cuda.Stream()
    kc = torch.empty((L, w.batch, w.num_kv_heads, 1, w.head_dim), dtype=torch.float16, device="cuda")
    vc = torch.empty_like(kc)
    qc = torch.empty((L, w.batch, w.num_q_heads, w.head_dim), dtype=torch.float16, device="cuda")
    out = torch.empty((L, w.batch, w.num_q_heads, w.head_dim), device="cuda")
    steps = 100  # crosses flushes of every layer and shrinks the RPC windows
    ins = []
    for s in range(steps):
        ks, vs = zip(*(W.gen_kv(w, l, w.context + s, 1, device="cuda") for l in range(L)))
        ins.append((torch.stack(ks), torch.stack(vs), torch.stack([W.gen_q(w, l, s, device="cuda") for l in range(L)])))
    torch.cuda.synchronize()

    def run():
        res = []
        with torch.cuda.stream(stream):
            for s in range(steps):
                kc.copy_(ins[s][0])
                vc.copy_(ins[s][1])
                qc.copy_(ins[s][2])
                c.decode_step([kc[l] for l in range(L)], [vc[l] for l in range(L)], [qc[l] for l in range(L)],
                              [out[l] for l in range(L)], stream=stream)
                res.append(out.clone())
        stream.synchronize()
        return res

    snap = c.save_state(stream=stream)
    v0 = _views(c, L)
    first = run()
    v1 = _views(c, L)
    assert v1 != v0
    c.restore_state(snap, stream=stream)
    assert _views(c, L) == v0
    second = run()
    assert _views(c, L) == v1
    for s in range(steps):
        assert torch.equal(first[s], second[s]), s
    assert c.device_error() == 0
    c.close()


def test_restore_mid_stream_multi_token_appends():
    w = _workload()
    L = w.num_layers
    c = _prefilled(w)
    sched = [1, 37, 1, 1, 64, 5, 1]
    inputs = []
    pos = w.context
    for n in sched:
        inputs.append([W.gen_kv(w, l, pos, n, device="cuda") for l in range(L)])
        pos += n
    qs = [W.gen_q(w, l, 7, device="cuda") for l in range(L)]

    def run(start):
        outs = []
        for i in range(start, len(sched)):
            for l in range(L):
                c.append(l, *inputs[i][l])
                outs.append(c.decode_attn(l, qs[l]).clone())
        return outs

    run_pre = run  # appends 0..1, then the snapshot
    for i in range(2):
        for l in range(L):
            c.append(l, *inputs[i][l])
    snap = torch.empty(K.kvq_state_bytes(c.h), dtype=torch.uint8, device="cuda")
    c.save_state(snap)
    a = run_pre(2)
    c.restore_state(snap)
    b = run_pre(2)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert c.device_error() == 0
    c.close()


def test_restore_refuses_unreachable_state():
    w = _workload()
    L = w.num_layers
    c = _prefilled(w)
    q = [W.gen_q(w, l, 0, device="cuda") for l in range(L)]
    before = [c.decode_attn(l, q[l]).clone() for l in range(L)]
    v0 = _views(c, L)
    bad = torch.zeros(K.kvq_state_bytes(c.h), dtype=torch.uint8, device="cuda")  # bound 0 < G
    with pytest.raises(K.KVQError) as e:
        c.restore_state(bad)
    assert e.value.status == 6
    assert _views(c, L) == v0
    after = [c.decode_attn(l, q[l]) for l in range(L)]
    for x, y in zip(before, after):
        assert torch.equal(x, y)
    # a snapshot from another handle of the same configuration is accepted
    other = _prefilled(w)
    snap = other.save_state()
    c.restore_state(snap)
    for l in range(L):
        assert torch.equal(c.decode_attn(l, q[l]), other.decode_attn(l, q[l]))
    assert c.device_error() == 0
    other.close()
    c.close()
