"""The KVQ_DEBUG build: every kernel range-checks its computed accesses
(records, rings, split partials, chunk workspace) against the buffers it was
given and reports a miss through the error word instead of touching memory
outside them.  A subset of the parity suite runs against the debug library
in a child process; each of those tests ends by requiring a clear error
word, so any check firing on a correct run fails it."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUBSET = ("test_stream_bitexact_and_attention or test_per_token_keys_bitexact or test_gqa_ratios or "
          "test_group_sizes or test_single_token or test_decode_step_graph or test_workload_tiny or "
          "test_chunk_all_pairs_d128 or test_chunk_window_only or test_chunk_after_single or "
          "test_chunk_gqa or test_noalloc")


def test_parity_subset_under_the_debug_build():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mixed_precision_quantized_quant_gb300 import build
    lib = build.build(debug=True)
    assert lib.endswith("libkvq_debug.so")
    env = dict(os.environ, KVQ_DEBUG_LIB="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
         "tests/test_gpu_parity.py", "tests/test_gpu_chunk.py", "tests/test_zz_no_alloc.py", "-k", SUBSET],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "deselected" in r.stdout, tail
