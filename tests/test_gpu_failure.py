"""Failure detection on the GPU without a fault: a device-side wait that
nothing completes gives up within its bound, reports the timeout through
the error word, and leaves the context usable for the next calls."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import kvq_oracle as O
from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import workloads as W
from tests.kvq_testutil import assert_attn_close

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    w = W.workload(1)
    kb, vb, R = w.layers[0][:3]
    cache = K.KVQCache(w.layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size, w.total_tokens)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        K.kvq_selftest_bounded_wait(cache.h, int(stream.cuda_stream))
        assert cache.device_error() == 0  # read and cleared by the self-test
    # the context still runs the real kernels correctly
    ora = O.OracleLayerCache(w.batch, w.num_kv_heads, w.head_dim, w.group_size, kb, vb, R)
    k, v = W.gen_kv(w, 0, 0, w.context, device="cuda")
    cache.append(0, k, v)
    ora.append(k.cpu().numpy(), v.cpu().numpy())
    q = W.gen_q(w, 0, 0, device="cuda")
    out = cache.decode_attn(0, q)
    torch.cuda.synchronize()
    assert_attn_close(out.cpu().numpy(), ora.attend(q.cpu().numpy()), "after the self-test")
    assert cache.device_error() == 0
    cache.close()
