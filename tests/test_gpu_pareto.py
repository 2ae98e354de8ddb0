"""Intra-layer pair pruning on the GPU (KVTuner A2, two-stage search-space
pruning, step 1): e_o per pair from the library's kernels against the
oracle's fp64 e_o, and the resulting Pareto front."""

from __future__ import annotations

import pytest

torch = pytest.importorskip("torch")

from oracle import kvq_oracle as O
from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import pareto as P
from mixed_precision_quantized_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# e_o is a mean of elementwise ratios |o - o_hat| / |o|.  The kernel's o_hat
# differs from the oracle's fp64 o_hat by at most the attention parity bound
# (2e-3 absolute, typically ~1e-5), and its exact-window o from the fp64 o by
# fp32 rounding.  Elements with a small |o| amplify both, hence a relative
# tolerance of a few percent on e_o itself.
E_RTOL = 0.03
E_ATOL = 1e-4


def _case(batch=1, hkv=2, hq=8, T=512, n_q=2, seed_layer=5, D=None, G=None):
    w = W.scaled(W.workload(2), batch=batch, num_kv_heads=hkv, num_q_heads=hq, context=T, decode_steps=n_q)
    if D is not None:
        w = W.scaled(w, head_dim=D)
    if G is not None:
        w = W.scaled(w, group_size=G)
    # drawn on the CPU, as in the oracle's pin of the same case, then moved
    k, v = (x.cuda() for x in W.gen_kv(w, seed_layer, 0, T))
    qs = [W.gen_q(w, seed_layer, s).cuda() for s in range(n_q)]
    return w, k, v, qs


def _check(gpu, ora):
    assert set(gpu) == set(ora)
    for p in ora:
        assert abs(gpu[p] - ora[p]) <= E_RTOL * ora[p] + E_ATOL, (p, gpu[p], ora[p])


def test_pair_errors_and_front_match_oracle():
    w, k, v, qs = _case()
    front, err = P.prune_layer_pairs(k, v, qs, P.ALL_PAIRS, w.group_size)
    ora = O.pair_output_errors(k.cpu().numpy(), v.cpu().numpy(), [q.cpu().numpy() for q in qs],
                               P.ALL_PAIRS, w.group_size, w.group_size)
    _check(err, ora)
    # over the {2, 4, 8}^2 candidates the front is the set the pruning keeps
    kivi = {p: err[p] for p in P.KIVI_PAIRS}
    assert P.pareto_front(kivi) == [(2, 2), (4, 2), (4, 4), (8, 4), (8, 8)]
    assert P.pareto_front(kivi) == O.pareto_front({p: ora[p] for p in P.KIVI_PAIRS})
    assert err[(4, 2)] < err[(2, 4)]


@pytest.mark.parametrize("D,G,gqa,R", [(64, 32, 1, 64), (128, 64, 7, 0), (128, 128, 4, 128)])
def test_pair_errors_shapes(D, G, gqa, R):
    w, k, v, qs = _case(batch=2, hkv=2, hq=2 * gqa, T=3 * G + 17, n_q=2, D=D, G=G)
    pairs = [(2, 2), (3, 3), (4, 2), (8, 4), (2, 8)]
    err = P.pair_output_errors(k, v, qs, pairs, w.group_size, R)
    ora = O.pair_output_errors(k.cpu().numpy(), v.cpu().numpy(), [q.cpu().numpy() for q in qs],
                               pairs, w.group_size, R or w.group_size)
    _check(err, ora)


def test_pair_errors_per_token_keys():
    w, k, v, qs = _case(T=384)
    err = P.pair_output_errors(k, v, qs, P.KIVI_PAIRS, w.group_size, 0, K.KEY_PER_TOKEN)
    ora = O.pair_output_errors(k.cpu().numpy(), v.cpu().numpy(), [q.cpu().numpy() for q in qs],
                               P.KIVI_PAIRS, w.group_size, w.group_size, O.KEY_PER_TOKEN)
    _check(err, ora)
    with pytest.raises(ValueError):
        P.pair_output_errors(k, v, qs, [(3, 2)], w.group_size, 0, K.KEY_PER_TOKEN)


def test_exact_window_reference_has_no_error():
    # a candidate whose window holds every token computes the reference's
    # attention; only the split of the sum over CTAs may differ
    w, k, v, qs = _case(T=200)
    err = P.pair_output_errors(k, v, qs, [(2, 2)], w.group_size, w.group_size * 7)
    assert err[(2, 2)] < 1e-5
