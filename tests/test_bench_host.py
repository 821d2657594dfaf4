"""Host-side logic of the benchmark that needs no GPU: the clock summary over
in-process samples, the roofline denominators and the check that refuses a
kernel far above its measured peak."""
import pytest

import bench


class _Dev:
    index = 0


def test_clock_summary_of_samples():
    c = bench.Clocks.__new__(bench.Clocks)
    c.samples = [(2070, [], 900.0), (1800, ["sw_power_cap"], 1400.0), (1750, ["sw_power_cap"], 1399.0),
                 (300, [], 100.0), (None, None, None)]
    c.max_mhz = 2070
    c.errors = []
    c.source = "nvml"
    c.nvml = object()
    c.period = 0.002
    s = c.summary()
    # the idle sample (below half the maximum) stays out of the median
    assert s["samples"] == 4 and s["sm_mhz"] == 1800 and s["sm_mhz_min"] == 1750
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1400.0
    assert s["source"] == "nvml" and s["period_ms"] == 2.0


def test_peaks_are_burst_figures_and_fp8_doubles_bf16():
    pk = bench.peaks()
    assert bench.tensor_peak(pk, fp8=False) == pk["bf16"]
    assert bench.tensor_peak(pk, fp8=True) == 2.0 * pk["bf16"]


def test_fraction_far_above_peak_is_refused():
    assert bench.check_frac("k", 1.04) == 1.04
    with pytest.raises(RuntimeError):
        bench.check_frac("k", 1.8)


def test_algorithmic_bytes_of_the_large_gemms():
    # FP8: A8 + B8 + bf16 C; INT8: qa + qb + fp32 C (codes read once, output written once)
    assert bench.algo_bytes("gemm_fp8_nt") == 469_762_048
    assert bench.algo_bytes("gemm_i8_kernel") == 738_197_504
