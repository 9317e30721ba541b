"""Host-side pieces of bench.py: the clock sampler's reading of nvidia-smi
lines (which trail the GPU's state) and the choice of the tensor peak for
the roofline (burst, or sustained when the timed region ran power-capped)."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def line(mhz, capped=False, hw=False):
    a = "Active" if capped else "Not Active"
    h = "Active" if hw else "Not Active"
    return f"{mhz}, 2070, 900.0, 0x{4 if capped else 0:016x}, {h}, Not Active, Not Active, {a}"


def sampler_with(samples):
    s = bench.ClockSampler(0)
    s.samples = samples
    return s


def test_cap_reported_after_the_region_is_still_counted():
    # the region is [10, 10.2]; the reading that shows the cap comes 0.2 s late
    s = sampler_with([(9.9, line(2070)), (10.05, line(2070)), (10.15, line(2070)),
                      (10.25, line(2070)), (10.4, line(1525, capped=True)), (11.0, line(2070))])
    c = s.summary(10.0, 10.2)
    assert c["reasons"] == ["sw_power_cap"]
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070


def test_clock_median_from_the_lagged_window():
    samples = [(10.0 + 0.02 * i, line(1525 if i >= 5 else 2070, capped=i >= 5)) for i in range(20)]
    c = sampler_with(samples).summary(10.0, 10.3)
    # readings between 10.1 and 10.4: all after the drop
    assert c["sm_mhz"] == 1525 and "sw_power_cap" in c["reasons"]


def test_no_reason_when_nothing_throttles():
    samples = [(10.0 + 0.02 * i, line(2070)) for i in range(30)]
    c = sampler_with(samples).summary(10.0, 10.3)
    assert c["reasons"] == [] and c["sm_mhz"] == 2070


def test_hw_slowdown_is_reported():
    samples = [(10.0 + 0.02 * i, line(2070, hw=(i == 7))) for i in range(30)]
    assert "hw_slowdown" in sampler_with(samples).summary(10.0, 10.3)["reasons"]


def test_peak_follows_the_regime():
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        peaks = json.load(f)
    flops, abytes, ms = 2 * 8192 ** 3, 8192 * 8192 * 8, 0.7
    burst = bench.roofline_of(flops, abytes, ms, None, "k",
                              {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    capped = bench.roofline_of(flops, abytes, ms, None, "k",
                               {"sm_mhz": 1525.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    low_clock = bench.roofline_of(flops, abytes, ms, None, "k",
                                  {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert burst["bound"] == "tensor" and burst["peak"] == peaks["bf16_tflops"]
    assert capped["peak"] == peaks["bf16_tflops_sustained"] == low_clock["peak"]
    assert capped["frac"] == pytest.approx(capped["achieved"] / peaks["bf16_tflops_sustained"], abs=1e-4)
    assert "sustained" in capped["peak_source"] and "burst" in burst["peak_source"]
    # a bandwidth-bound launch keeps the copy bandwidth whatever the clocks
    hbm = bench.roofline_of(2 * 256 * 256 * 65536, 67 * 2 ** 20, 0.027, None, "k",
                            {"sm_mhz": 1525.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    assert hbm["bound"] == "hbm" and hbm["peak"] == peaks["hbm_gbs"]


def test_burst_object_uses_the_burst_peak():
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        peaks = json.load(f)
    flops = 2 * 8192 ** 3
    bo = bench.burst_of(flops, 8192 * 8192 * 8, 0.655)
    assert bo["steps"] == 30 and bo["bound"] == "tensor" and bo["peak"] == peaks["bf16_tflops"]
    assert bo["value"] == pytest.approx(flops / 0.655e-3 / 1e12, rel=1e-4)
    assert bo["roofline_frac"] == pytest.approx(bo["value"] / peaks["bf16_tflops"], abs=1e-4)
    # a bandwidth-bound shape against the copy bandwidth
    lk = bench.burst_of(2 * 256 * 256 * 65536, 67 * 2 ** 20, 0.027)
    assert lk["bound"] == "hbm" and lk["peak"] == peaks["hbm_gbs"]


def test_per_clock_peak():
    # 152 SMs x 8192 flop/clk: 2577.5 TFLOP/s at 2070 MHz, 1869.7 at 1501.5 MHz
    r = bench.per_clock_peak(1400.0, {"sm_mhz": 1501.5, "sm_max_mhz": 2070.0}, sms=152)
    assert r["flop_per_clk_per_sm"] == 8192 and r["sms"] == 152
    assert r["at_max_clock"]["tflops"] == round(152 * 8192 * 2070e6 / 1e12, 1)
    assert abs(r["at_max_clock"]["frac"] - 1400.0 / (152 * 8192 * 2070e6 / 1e12)) < 1e-4
    assert abs(r["at_load_clock"]["frac"] - 1400.0 / (152 * 8192 * 1501.5e6 / 1e12)) < 1e-4
    # no clocks: only the SM count and rate
    assert set(bench.per_clock_peak(1.0, None, sms=4)) == {"sms", "flop_per_clk_per_sm"}
