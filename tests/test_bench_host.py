"""Host logic of bench.py on CPU: the clock record's summary (throttle reasons,
median SM clock), the roofline arithmetic and the choice of its bound, and the
rule that a committed ncu traffic figure is reported only while the source it
was captured from is unchanged."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _sampler(lines):
    import bench
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.lines = lines
    s.err = ""
    return s


def test_clock_summary_reasons_and_median():
    lines = ["1900, 2032, 700.1, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2032, 2032, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
             "2000, 2032, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
             "garbage line"]
    out = _sampler(lines).summary()
    assert out["sm_mhz"] == 2000.0 and out["sm_max_mhz"] == 2032.0 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    hot = _sampler(["1500, 2032, 1000, 0x48, Active, Active, Not Active, Not Active"]).summary()
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clock_summary_without_samples():
    out = _sampler([]).summary()
    assert out["samples"] == 0 and out["reasons"] == ["unsampled"] and out["sm_mhz"] is None


PEAKS = {"hbm_gbs": 1000.0, "source": "measured"}
PIPES = {"ex2": {"ops_per_s": 4e12}, "ffma2": {"ops_per_s": 16e12}}


def test_roofline_terms_and_bound():
    import bench
    # 1e9 elements x N 16 in 10 ms: 1.6e12 ex2/s (40% of 4e12), 6.4e12 fp32/s (40% of 16e12),
    # 5e9 bytes: 500 GB/s (50% of 1000): HBM is the bound
    r = bench.roofline_s6(1e9, 16, 5e9, 10.0, PEAKS, PIPES)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(500.0) and r["frac"] == pytest.approx(0.5)
    assert r["terms"]["sfu"]["frac"] == pytest.approx(0.4) and r["terms"]["fp32"]["frac"] == pytest.approx(0.4)
    assert r["traffic"] is None and r["algorithmic_bytes"] == 5e9
    # fewer bytes: the ALU terms bound it, and the larger of them is reported
    r = bench.roofline_s6(1e9, 16, 1e9, 10.0, PEAKS, PIPES, exps_per_elem_n=1.5)
    assert r["bound"] == "alu" and r["unit"] == "Gex2/s" and r["frac"] == pytest.approx(0.6)


def test_traffic_only_for_the_captured_source(tmp_path):
    import bench
    assert bench._ncu_traffic("no_such_kernel", __file__) is None
    assert bench._ncu_traffic("conv1d_fwd_w4_kernel", str(tmp_path / "missing.cu")) is None
    src = tmp_path / "k.cu"
    src.write_text("// one version of a kernel\n")
    sha = bench._sha(str(src))
    saved = dict(bench.NCU_TRAFFIC)
    try:
        bench.NCU_TRAFFIC["k_kernel"] = {"src_sha": sha, "bytes_per_launch": 123.0}
        assert bench._ncu_traffic("k_kernel", str(src)) == 123.0
        r = bench.roofline_s6(1e6, 16, 1e6, 1.0, PEAKS, PIPES, kernel="k_kernel", src=str(src))
        assert r["traffic"] == 123.0
        src.write_text("// the kernel, changed after the capture\n")
        assert bench._ncu_traffic("k_kernel", str(src)) is None
        r = bench.roofline_s6(1e6, 16, 1e6, 1.0, PEAKS, PIPES, kernel="k_kernel", src=str(src))
        assert r["traffic"] is None
    finally:
        bench.NCU_TRAFFIC.clear()
        bench.NCU_TRAFFIC.update(saved)


def test_whole_job_rate_is_weak_scaling():
    import bench
    # 1000 units per rank and step, 5 steps, slowest rank 10 ms
    assert bench.whole_job_rate(1000, 5, 1, 10.0) == pytest.approx(5e5)
    assert bench.whole_job_rate(1000, 5, 8, 10.0) == pytest.approx(4e6)
