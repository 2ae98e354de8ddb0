"""kvq_decode_attn_noalloc: the decode entry point for callers that may not
allocate device memory (a plugin whose host runtime owns every allocation, or
a latency path where a synchronising cudaMalloc is not allowed).  Its
split-merge workspace lives in the library's static device array, so this
file checks that it gives the same attention as kvq_decode_attn on two calls
in a row (the second one finds the array as the first left it), and that a
layer needing more workspace than the array holds is refused.

Kept in a file of its own, collected after the other GPU tests."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import workloads as W
from tests.kvq_testutil import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    K.load()


def _noalloc(cache, layer, q, out, stream):
    K.kvq_decode_attn_noalloc(cache.h, layer, int(q.data_ptr()), int(out.data_ptr()), stream.cuda_stream)


def test_noalloc_matches_decode_attn_twice():
    # few (batch, kv head) units over a long context: every unit is split over
    # many CTAs, so the merge goes through the workspace
    w = W.scaled(W.workload(2), batch=2, num_layers=2, context=3000, decode_steps=4,
                 layers=((8, 4, 32), (4, 2, 32)))
    cache = K.KVQCache(w.layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size,
                       w.total_tokens)
    stream = torch.cuda.Stream()
    for l in range(w.num_layers):
        k, v = W.gen_kv(w, l, 0, w.context, device="cuda")
        cache.append(l, k, v)
    torch.cuda.synchronize()
    shape = (w.batch, w.num_q_heads, w.head_dim)
    for step in range(2):
        for l in range(w.num_layers):
            k, v = W.gen_kv(w, l, w.context + step, 1, device="cuda")
            q = W.gen_q(w, l, step, device="cuda")
            ref = torch.empty(shape, dtype=torch.float32, device="cuda")
            got = [torch.full(shape, float("nan"), device="cuda") for _ in range(2)]
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                cache.append(l, k, v, stream=stream)
                cache.decode_attn(l, q, ref, stream=stream)
                for g in got:  # two calls in a row on the same state
                    _noalloc(cache, l, q, g, stream)
            stream.synchronize()
            r = ref.cpu().numpy()
            for i, g in enumerate(got):
                assert_attn_close(g.cpu().numpy(), r, f"step {step} layer {l} call {i}")
    assert cache.device_error() == 0
    cache.close()


def test_noalloc_rejects_oversized_workspace():
    # 1024 units x gqa 8 x (128 + 2) floats per split slot exceed the 4 MiB array
    cache = K.KVQCache([(4, 2, 32)], 128, 64, 8, 128, 32, 64)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    k = torch.randn((128, 8, 4, 128), generator=gen, device="cuda").half()
    cache.append(0, k, k)
    q = torch.randn((128, 64, 128), generator=gen, device="cuda").half()
    out = torch.zeros((128, 64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(K.KVQError) as ei:
        _noalloc(cache, 0, q, out, torch.cuda.current_stream())
    assert ei.value.status == 4  # KVQ_ERR_CAPACITY
    torch.cuda.synchronize()
    assert not out.any()  # nothing was launched
    cache.close()
