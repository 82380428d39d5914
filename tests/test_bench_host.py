"""Host-side logic of bench.py, on the CPU: the roofline of a pass, the
whole-job rate over ranks, the committed DRAM-traffic lookup (valid only for
the kernel sources it was measured on), the measured-peaks file with its
fallback, and the clock sampler's summary of nvidia-smi rows."""
from __future__ import annotations

import json

import pytest

import bench

PK = {"bf16_tflops": 1890.9, "hbm_gbs": 6759.9}


def test_roofline_memory_bound_pass():
    # fp16 7x7 forward: 154.2 MB unique in 49.5 us, 3.55 GFLOP valid on the tensor cores.
    r = bench.pass_roofline("tiled_mma", 3.5488e9, 154.16e6, 0.0495, PK, 80.55)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(154.16e6 / 49.5e-6 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx((154.16e6 / 6759.9e9) / 49.5e-6, rel=1e-3)


def test_roofline_compute_bound_passes_take_their_own_unit():
    # A CUDA-core pass is held against the FMA peak, a tensor-core pass against the bf16 peak.
    alu = bench.pass_roofline("tiled_wgrad", 3.5488e9, 154.16e6, 0.0822, PK, 80.55)
    assert alu["bound"] == "alu" and alu["peak"] == 80.55
    assert alu["frac"] == pytest.approx(3.5488e9 / 80.55e12 / 82.2e-6, rel=1e-3)
    ten = bench.pass_roofline("tiled_mma_large", 18.33e9, 51.6e6, 0.118, PK, 80.55)
    assert ten["bound"] == "tensor" and ten["peak"] == 1890.9
    assert ten["achieved"] == pytest.approx(18.33e9 / 0.118e-3 / 1e12, rel=1e-3)


def test_whole_job_rate_counts_every_rank_over_the_slowest_time():
    one = bench.whole_job_rate(1, 11.3e9, 0.18)
    assert one == pytest.approx(11.3e9 / 0.18e-3 / 1e9)
    assert bench.whole_job_rate(4, 11.3e9, 0.18) == pytest.approx(4 * one)


def test_max_over_ranks_is_the_value_on_one_rank():
    assert bench.max_over_ranks(0.123, 1, "cpu") == 0.123


def test_recorded_traffic_only_for_the_sources_it_was_measured_on(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic_w.txt").write_text(
        "# comment = ignored\ncsrc_sha = abcdef0123456789\nfwd_dram_bytes = 130067968  # per launch\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "csrc_sha", lambda: "abcdef0123456789")
    assert bench.recorded_traffic("w", "fwd") == 130067968.0
    assert bench.recorded_traffic("w", "wgrad") is None
    assert bench.recorded_traffic("no-such-workload", "fwd") is None
    monkeypatch.setattr(bench, "csrc_sha", lambda: "0000000000000000")  # kernels changed since
    assert bench.recorded_traffic("w", "fwd") is None


def test_committed_traffic_is_near_the_unique_bytes_when_current():
    v = bench.recorded_traffic("fp16-train-7x7-128x56x56x96", "wgrad")
    if v is None:
        pytest.skip("kernel sources changed since the committed ncu capture")
    # x and dy (77 MB each) are read once: the recorded DRAM bytes are near that.
    assert 0.9 * 154.16e6 < v < 1.2 * 154.16e6


def test_csrc_sha_follows_the_kernel_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "depthwise_convolution_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("kernel a\n")
    (csrc / "b.cuh").write_text("header b\n")
    (csrc / "notes.txt").write_text("not a source\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    first = bench.csrc_sha()
    (csrc / "notes.txt").write_text("changed, still not a source\n")
    assert bench.csrc_sha() == first
    (csrc / "a.cu").write_text("kernel a, changed\n")
    assert bench.csrc_sha() != first


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.peaks()
    assert pk["source"] == "fallback" and pk["hbm_gbs"] == 6800.0 and pk["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6759.9, "bf16_tflops": 1890.9}))
    pk = bench.peaks()
    assert pk["source"] == "measured" and pk["hbm_gbs"] == 6759.9 and pk["bf16_tflops"] == 1890.9


def _row(sm, reasons=("Not Active",) * 4):
    return [str(sm), "2070", "900.0", *reasons]


def test_clock_summary_takes_the_median_inside_the_window_and_names_throttling():
    c = bench.ClockSampler(0)
    c.samples = [(0.5, _row(1200)),
                 (1.0, _row(2070)), (1.2, _row(2055)),
                 (1.4, _row(2070, ("Not Active", "Not Active", "Not Active", "Active"))),
                 (9.0, _row(300))]
    s = c.summary(1.0, 2.0)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    hot = bench.ClockSampler(0)
    hot.samples = [(1.0, _row(1500, ("Active", "Not Active", "Active", "Not Active")))]
    assert hot.summary(0.0, 2.0)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples_says_so():
    s = bench.ClockSampler(0).summary(0.0, 1.0)
    assert s["sm_mhz"] is None and s["reasons"] == ["no nvidia-smi samples"]
