"""The C-ABI library: it loads, exports every entry point include/kvq.h
declares, and its host-only sizing logic behaves.  No GPU needed."""

import ctypes
import os
import re

import pytest

from mixed_precision_quantized_quant_gb300 import kvq as K
from mixed_precision_quantized_quant_gb300 import workloads as W
from oracle import kvq_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(K.LIB_PATH):
        from mixed_precision_quantized_quant_gb300 import build
        build.build()
    return K.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(K.EXPORTS) == set(names), (set(K.EXPORTS) ^ set(names))
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(8):
        assert K.kvq_status_string(code)
    assert K.kvq_status_string(0) == "ok"


def _cfg(**kw):
    base = dict(layers=[(4, 2, 32)], batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=32,
                max_tokens=1024)
    base.update(kw)
    return K.make_config(base.pop("layers"), **base)


def test_cache_bytes_rejects_bad_configs(lib):
    assert K.kvq_cache_bytes(_cfg()) > 0
    bad = [dict(head_dim=96), dict(group_size=48), dict(num_q_heads=6, num_kv_heads=4),
           dict(num_q_heads=32, num_kv_heads=2), dict(layers=[(5, 2, 32)]), dict(layers=[(4, 2, 48)]),
           dict(layers=[(4, 2, 16)]), dict(batch=0), dict(max_tokens=0),
           dict(layers=[(3, 2, 32, 1)]), dict(layers=[(4, 2, 32, 2)]), dict(layers=[(4, 2, 32, 0, 101)])]
    for b in bad:
        assert K.kvq_cache_bytes(_cfg(**b)) == 0, b


def test_cache_bytes_covers_layout(lib):
    # the buffer holds at least the records for max_tokens and the windows
    for idx in range(1, 7):
        w = W.workload(idx)
        cfg = K.make_config(w.layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size,
                            w.total_tokens)
        nb = K.kvq_cache_bytes(cfg)
        U = w.batch * w.num_kv_heads
        need = 0
        for kb, vb, R, _, _ in map(W.spec_fields, w.layers):
            rec = O.record_layout(w.head_dim, w.group_size, kb, vb)["bytes"]
            need += U * (w.total_tokens // w.group_size) * rec + 2 * U * R * w.head_dim * 2
        assert need <= nb <= need * 1.02 + (64 << 20), (idx, nb, need)


def test_create_rejects_without_buffer(lib):
    h = ctypes.c_void_p()
    cfg = _cfg()
    st = lib.kvq_create(ctypes.byref(cfg), None, 0, ctypes.byref(h))
    assert st == 1 and not h.value
    st = lib.kvq_create(ctypes.byref(cfg), ctypes.c_void_p(256), 16, ctypes.byref(h))
    assert st == 4 and not h.value  # buffer too small: checked before any CUDA call
    st = lib.kvq_create(ctypes.byref(cfg), ctypes.c_void_p(8), 1 << 40, ctypes.byref(h))
    assert st == 3 and not h.value  # misaligned


def test_null_handle_calls_are_rejected(lib):
    assert lib.kvq_append(None, 0, None, None, 1, None) == 1
    assert lib.kvq_decode_attn(None, 0, None, None, None) == 1
    assert lib.kvq_destroy(None) == 1
    assert lib.kvq_equivalent_bits(None) == 0.0
    assert lib.kvq_decode_bytes(None, 0) == -1
    assert lib.kvq_state_bytes(None) == 0
    assert lib.kvq_state_save(None, None, None) == 1
    assert lib.kvq_state_restore(None, None, None) == 1


def test_per_token_key_layout(lib):
    # per-token keys: the record keeps one (scale, zero) pair per token for the keys
    for kb in (2, 4, 8):
        for vb in (2, 3, 4, 8):
            cfg = _cfg(layers=[(kb, vb, 32, 1)], max_tokens=64)
            assert K.kvq_cache_bytes(cfg) > 0
            lay = O.record_layout(128, 32, kb, vb, O.KEY_PER_TOKEN)
            lay0 = O.record_layout(128, 32, kb, vb)
            assert lay["bytes"] == lay0["bytes"] - 4 * 128 + 4 * 32


def test_rpc_ratio_accepted_up_to_100(lib):
    for pct in (0, 1, 10, 20, 100):
        assert K.kvq_cache_bytes(_cfg(layers=[(4, 2, 160, 0, pct)])) > 0


def test_binding_structs_match_the_header(tmp_path):
    # sizes and field offsets of the public structs as a C compiler lays them
    # out from include/kvq.h, against the ctypes mirrors in the binding
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"kvq_layer_cfg": K.LayerCfg, "kvq_layer_view": K.LayerView, "kvq_config": K.Config}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "kvq.h"', "int main(void) {"]
    for cname, py in fields.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("  return 0;\n}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l}
    for cname, py in fields.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)
