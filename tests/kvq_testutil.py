"""Helpers for the GPU parity tests: read the device cache back in the
documented layout and drive the oracle on the same fp16 inputs."""

from __future__ import annotations

import numpy as np

from oracle import kvq_oracle as O

ATOL = 2e-3      # max-abs attention error against fp64 over the same dequantized values
RTOL_L2 = 1e-3   # relative L2 error


def buf_slice(cache, ptr: int, nbytes: int) -> np.ndarray:
    base = int(cache.buf.data_ptr())
    off = ptr - base
    return cache.buf[off:off + nbytes].cpu().numpy()


def gpu_unit_records(cache, layer: int, u: int) -> bytes:
    v = cache.view(layer)
    n = (v["quantized_tokens"] // v["group_size"]) * v["record_bytes"]
    return buf_slice(cache, v["records"] + u * v["unit_record_stride"], n).tobytes()


def gpu_unit_ring(cache, layer: int, u: int):
    """Ring contents [R, D] fp16 for K and V with the chunk swizzle undone."""
    v = cache.view(layer)
    R, D = v["residual"], v["head_dim"]
    out = []
    for key in ("residual_k", "residual_v"):
        raw = buf_slice(cache, v[key] + u * v["residual_stride"], R * D * 2).view(np.float16).reshape(R, D // 8, 8)
        nat = np.empty_like(raw)
        for s in range(R):
            for c in range(D // 8):
                nat[s, c] = raw[s, c ^ (s & 7)]
        out.append(nat.reshape(R, D))
    return out[0], out[1]


def compare_layer(cache, layer: int, ora: O.OracleLayerCache, units=None) -> None:
    """Bit-exact comparison of group records and live ring slots."""
    v = cache.view(layer)
    assert v["tokens"] == ora.total
    assert v["quantized_tokens"] == ora.n_q and v["residual_tokens"] == ora.r
    if units is None:
        units = range(ora.B * ora.H)
    live = ora.live_ring_slots()
    for u in units:
        got = gpu_unit_records(cache, layer, u)
        exp = ora.unit_records(u)
        if got != exp:
            raise AssertionError(describe_record_mismatch(got, exp, ora, u))
        if len(live):
            gk, gv = gpu_unit_ring(cache, layer, u)
            ok_, ov_ = ora.residual_ring(u)
            assert np.array_equal(gk[live].view(np.uint16), ok_[live].view(np.uint16)), f"ring K unit {u}"
            assert np.array_equal(gv[live].view(np.uint16), ov_[live].view(np.uint16)), f"ring V unit {u}"


def describe_record_mismatch(got: bytes, exp: bytes, ora, u: int) -> str:
    lay = O.record_layout(ora.d, ora.G, ora.kb, ora.vb, ora.key_mode)
    rb = lay["bytes"]
    if len(got) != len(exp):
        return f"unit {u}: record bytes {len(got)} != {len(exp)}"
    g = np.frombuffer(got, np.uint8)
    e = np.frombuffer(exp, np.uint8)
    bad = np.nonzero(g != e)[0]
    first = int(bad[0])
    grp, off = divmod(first, rb)
    region = max((lay[k], k) for k in ("k_codes", "v_codes", "k_scale", "k_zero", "v_scale") if lay[k] <= off)[1]
    return (f"unit {u}: {len(bad)} bytes differ; first at group {grp} offset {off} ({region}); "
            f"got {g[first:first + 8].tolist()} expected {e[first:first + 8].tolist()}")


def attn_errors(got: np.ndarray, exp: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    exp = np.asarray(exp, dtype=np.float64)
    mx = float(np.abs(got - exp).max())
    rel = float(np.linalg.norm(got - exp) / max(np.linalg.norm(exp), 1e-30))
    return mx, rel


def assert_attn_close(got, exp, what=""):
    mx, rel = attn_errors(got, exp)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert mx <= ATOL and rel <= RTOL_L2, f"{what}: max-abs {mx:.3e}, rel-L2 {rel:.3e}"
