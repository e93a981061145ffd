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
