"""bench.py's host-side helpers (no GPU): the clock/throttle summary that
decides whether a run is kept, and the roofline fractions added to the sweep."""

import os
import sys

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), ".."))

import bench  # noqa: E402


def _row(sm, smax, power, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    # timestamp, index, clocks.sm, clocks.max.sm, power.draw, active mask, 4 reasons
    return ["2026/12/02 10:00:00.000", "0", str(sm), str(smax), str(power), "0x0", hw, hw_th, sw_th, cap]


def test_clock_summary_median_max_and_reasons():
    rows = [_row(2070, 2070, 400.5), _row(2055, 2070, 410.0), _row(2070, 2070, 420.0, cap="Active")]
    s = bench.ClockSampler.summarize(rows)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_median"] == 410.0


def test_clock_summary_flags_every_slowdown_reason():
    rows = [_row(1500, 2070, 300, hw="Active"), _row(1500, 2070, 300, hw_th="Active"),
            _row(1500, 2070, 300, sw_th="Active")]
    s = bench.ClockSampler.summarize(rows)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1500.0


def test_clock_summary_without_samples():
    s = bench.ClockSampler.summarize([])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["no samples"]


def test_sweep_fractions_use_the_measured_peaks():
    hbm, tflops, _ = bench.measured_peaks()
    node = {"a": {"us_per_call": 1.0, "weight_GBps": hbm / 2, "TOPS": tflops / 4},
            "b": {"1": {"gemv": {"weight_GBps": hbm}}, "fused_weight_GBps": hbm / 4}}
    bench._add_fractions(node)
    assert abs(node["a"]["frac_copy_bw"] - 0.5) < 1e-12
    assert abs(node["a"]["frac_bf16_peak"] - 0.25) < 1e-12
    assert abs(node["b"]["1"]["gemv"]["frac_copy_bw"] - 1.0) < 1e-12
    assert abs(node["b"]["fused_frac_copy_bw"] - 0.25) < 1e-12


def test_sweep_fractions_include_the_s8_peak():
    node = {"a": {"TOPS": bench.s8_peak_tops()}, "cpu_baseline": {"weight_GBps": 1.0}}
    bench._add_fractions(node)
    assert abs(node["a"]["frac_s8_peak"] - 1.0) < 1e-12
    assert "frac_copy_bw" not in node["cpu_baseline"]   # the oracle's own figures stay as they are


def test_s8_peak_from_the_measured_rate():
    # 223 MACs per clock per SM, 2 operations per MAC, 152 SMs, at 2070 MHz
    assert abs(bench.s8_peak_tops(2070.0) - 2 * 223 * 152 * 2070e6 / 1e12) < 1e-9


def test_oracle_baseline_of_a_sweep_row():
    """A sweep row's CPU baseline: the oracle's sampled work timed on one core,
    the rate per weight byte, the estimate for the whole call, the speed-up."""
    import numpy as np
    import qmm_synth
    N, K, g = 256, 256, 64
    lay = qmm_synth.Layer("bench_host", 0, N, K, g, g)
    qb, sw, _ = qmm_synth.layer_weights(0, "bench_host", lay)
    x = qmm_synth.layer_activations(0, "bench_host", lay, 2)
    rows = bench._sample_rows(N, 16)
    per_row = K // 2 + 2 * (K // g)
    task = {"kind": "w4a8", "x": x, "group": g, "had": g, "mats": [(qb[rows], sw[rows])],
            "bytes": rows.size * per_row, "ops": 2 * 2 * rows.size * K, "full_bytes": N * per_row,
            "sample": "test"}
    row = {"weight_GBps": 100.0}
    bench.oracle_baselines([(row, task)], None, seconds=0.05)
    base = row["cpu_baseline"]
    assert base["kind"] == "oracle" and base["cores"] == 1 and base["sample"] == "test"
    assert base["weight_GBps"] > 0 and base["GOPS"] > 0
    assert abs(base["us_per_call_est"] - N * per_row / (base["weight_GBps"] * 1e9) * 1e6) < 1e-6
    assert abs(base["gpu_speedup_vs_1_core"] - 100.0 / base["weight_GBps"]) < 1e-9
    assert np.isfinite(base["us_per_call_est"])
    # the same figures flat on the row
    assert row["oracle_us"] == base["us_per_call_est"] and row["oracle_GBps"] == base["weight_GBps"]
    assert row["oracle_cores"] == 1 and "oracle_all_cores" not in row
