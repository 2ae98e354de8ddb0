"""Host logic of the pair-pruning tool: its Pareto filter against the
oracle's on random error tables, and its argument checks (no GPU)."""

from __future__ import annotations

import random

import pytest

from oracle import kvq_oracle as O
from mixed_precision_quantized_quant_gb300 import pareto as P


def test_front_matches_oracle_filter_on_random_tables():
    rng = random.Random(7)
    for trial in range(200):
        pairs = rng.sample(list(P.ALL_PAIRS), rng.randint(1, 16))
        # coarse values so that ties in e_o happen
        err = {p: rng.choice([0.001, 0.01, 0.02, 0.05, 0.1, 0.2]) for p in pairs}
        got = P.pareto_front(err)
        exp = O.pareto_front(err)
        assert sorted(got) == sorted(exp), (trial, err)
        # cheapest first; along the front e_o strictly falls as bits rise
        bits = [P.equivalent_bits(p) for p in got]
        assert bits == sorted(bits)
        for a, b in zip(got, got[1:]):
            if P.equivalent_bits(a) < P.equivalent_bits(b):
                assert err[b] < err[a]


def test_candidate_sets():
    assert len(P.ALL_PAIRS) == 16 and len(P.KIVI_PAIRS) == 9
    assert set(P.KIVI_PAIRS) <= set(P.ALL_PAIRS)
    assert P.equivalent_bits((8, 4)) == 6.0


def test_rejects_empty_queries_before_touching_a_device():
    with pytest.raises(ValueError):
        P.pair_output_errors(None, None, [])
