"""Host-side logic of bench.py, on CPU: the chunk FLOP count against a brute
count of visible (query, key) pairs, the clock-sample summary (median SM
clock, throttle reasons seen inside the timed windows), the lookup of the
committed DRAM-traffic figure (only while the decode source it was taken on
is unchanged), and the peak denominators with and without the measured-peaks
file."""

import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("B,Hq,D,T,n", [(1, 1, 1, 1, 1), (1, 2, 4, 7, 3), (2, 3, 8, 10, 10), (1, 1, 16, 33, 1)])
def test_chunk_flops_counts_visible_pairs(B, Hq, D, T, n):
    # query i sits at position T - n + i and sees positions 0 .. T - n + i
    visible = sum(T - n + i + 1 for i in range(n))
    assert bench._chunk_flops(B, Hq, D, T, n) == 4.0 * D * visible * Hq * B


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _line(sm, smax, slowdown="Not Active", power_cap="Not Active"):
    # index, timestamp, clocks.sm, clocks.max.sm, power, active mask, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return f"0, 2026/01/01 00:00:00.000, {sm}, {smax}, 900.0, 0x0, {slowdown}, Not Active, Not Active, {power_cap}"


def test_clock_summary_uses_the_timed_windows():
    s = bench.ClockSampler(0)
    s._proc = _DoneProc()
    s.samples = [(1.0, _line(1000, 2070, slowdown="Active")),   # before the window: ignored
                 (10.0, _line(2070, 2070)),
                 (10.5, _line(2055, 2070, power_cap="Active")),
                 (11.0, _line(2070, 2070)),
                 (20.0, _line(500, 2070, slowdown="Active"))]   # after it: ignored
    s.mark(10.0, 11.0)
    c = s.stop()
    assert c["in_timed_region"] is True
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2070.0
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples_in_window_uses_all():
    s = bench.ClockSampler(0)
    s._proc = _DoneProc()
    s.samples = [(1.0, _line(1900, 2070, slowdown="Active")), (2.0, _line(2000, 2070))]
    s.mark(50.0, 51.0)
    c = s.stop()
    assert c["in_timed_region"] is False
    assert c["samples"] == 2
    assert c["sm_mhz"] == 1950.0
    assert c["reasons"] == ["hw_slowdown"]


def test_clock_summary_without_nvidia_smi():
    s = bench.ClockSampler(0)
    assert s.stop() is None


def _fake_tree(tmp_path, source, recorded_sha):
    csrc = tmp_path / "mixed_precision_quantized_quant_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "kvq_decode.cuh").write_bytes(source)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "decode_kernel_dram_w.txt").write_text(
        "# summary\n\nworkload: w\n"
        f"kernel_source_sha256_16: {recorded_sha}\n"
        "dram_bytes_per_launch_mean: 70039784\n\n| table | row |\n")


def test_traffic_figure_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    src = b"// decode kernel source\n"
    sha = hashlib.sha256(src).hexdigest()[:16]
    _fake_tree(tmp_path, src, sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._ncu_traffic("w") == 70039784
    # the kernel changed since the capture: no figure
    (tmp_path / "mixed_precision_quantized_quant_gb300" / "csrc" / "kvq_decode.cuh").write_bytes(src + b"//\n")
    assert bench._ncu_traffic("w") is None
    # no capture for this workload
    assert bench._ncu_traffic("other") is None


def test_peaks_measured_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._peaks() == (6800.0, "fallback")
    assert bench._tensor_peak() == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6770.5, "bf16_tflops": 1890.1}))
    assert bench._peaks() == (6770.5, "measured")
    assert bench._tensor_peak() == (1890.1, "measured")


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("warm,steps", [(3, 1), (3, 2), (5, 20), (8, 120), (3, 300)])
def test_prefill_offset_puts_a_flush_of_every_layer_in_the_window(index, warm, steps):
    # the middle timed step quantizes a key group on every layer (flush rule
    # replayed by the oracle's token-by-token state machine)
    from mixed_precision_quantized_quant_gb300 import workloads as W
    from oracle import kvq_oracle as O
    w = W.workload(index)
    S0, mid = bench._prefill_length(w, warm, steps)
    assert warm < mid <= warm + steps
    assert 0 <= w.context - S0 < w.group_size
    for R in {spec[2] for spec in w.layers}:
        before, _ = O.flush_state(S0 + mid - 1, R, w.group_size)
        after, _ = O.flush_state(S0 + mid, R, w.group_size)
        assert after == before + w.group_size
