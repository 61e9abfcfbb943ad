"""Host-side logic of bench.py that needs no GPU: the one-GPU guard, the chip
peak arithmetic, kernel naming and the traffic lookup."""
import json
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from tensor_core_gemm_02_gb300 import binding, workloads  # noqa: E402


def test_more_than_one_gpu_is_refused(monkeypatch):
    """The bench runs on one GPU: --gpus 2, or a launch under torchrun with
    WORLD_SIZE 2, exits with status 2 before touching a GPU."""
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.single_gpu_only(1)  # the default passes
    with pytest.raises(SystemExit) as e:
        bench.single_gpu_only(2)
    assert e.value.code == 2
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit) as e:
        bench.single_gpu_only(1)
    assert e.value.code == 2


def test_spec_peak_from_sms_and_clock():
    """152 SMs x 8192 flop per clock at 2070 MHz is 2577.4 TFLOP/s; at a sampled
    median of 1650 MHz, 2054.5; the achieved rate is divided by each."""
    s = bench.spec_peak(152, {"sm_max_mhz": 2070.0, "sm_mhz": 1650.0}, 1800.0)
    assert s["peak_at_max_mhz"] == pytest.approx(152 * 8192 * 2.07e9 / 1e12, abs=0.06)
    assert s["peak_at_median_mhz"] == pytest.approx(152 * 8192 * 1.65e9 / 1e12, abs=0.06)
    assert s["frac_at_max_mhz"] == pytest.approx(1800.0 / (152 * 8192 * 2.07e9 / 1e12), abs=1e-4)
    assert s["frac_of_nominal"] == pytest.approx(1800.0 / 2250.0)  # the published dense figure
    assert s["frac_at_median_mhz"] == pytest.approx(1800.0 / (152 * 8192 * 1.65e9 / 1e12),
                                                    abs=1e-4)
    # no clock samples: no peak figures, no division
    assert "peak_at_median_mhz" not in bench.spec_peak(152, {"sm_mhz": None}, 1800.0)


def test_kernel_keys_name_the_launched_instance():
    binding.load_library()
    p = binding.gemm_query_plan(8192, 8192, 8192, e2m1=0, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 3, 0, 1, 1, 0, 1>"
    p = binding.gemm_query_plan(8192, 8192, 8192, e2m1=1, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 3, 0, 1, 1, 0, 2>"
    p = binding.gemm_query_plan(16, 28672, 4096, e2m1=0, sm_count=148)
    assert bench.kernel_key(p) == "skinny_gemm_kernel<16, 1, 0, 1>"
    p = binding.gemm_query_plan(8192, 8192, 8192, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 1, 2, 1, 0, 0>"
    p = binding.gemm_query_plan(8192, 28672, 4096, has_c=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 6, 1, 1, 1, 0, 0>"
    p = binding.gemm_query_plan(16, 28672, 4096, sm_count=148)
    assert bench.kernel_key(p) == "skinny_gemm_kernel<16, 1, 0, 0>"
    p = binding.gemm_query_plan(1024, 1024, 1024, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<64, 8, 0, 1, 1, 0, 0>"
    p = binding.gemm_query_plan(16384, 4096, 4096, gather=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 1, 2, 4, 0, 0>"
    p = binding.gemm_query_plan(16384, 1024, 4096, gather=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 1, 2, 2, 0, 0>"
    p = binding.gemm_query_plan(16384, 1024, 1024, gather=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 0, 1, 4, 0, 0>"
    # the epilogue mode and the FP4 converter warps come from the problem
    sc = workloads.Problem("s", torch.zeros(1, 1), torch.zeros(1, 1), idx=torch.zeros(1),
                           scatter=True, d_rows=1)
    p = binding.gemm_query_plan(16384, 4096, 4096, scatter=True, sm_count=148)
    assert bench.kernel_key(p, sc) == "tile_gemm_kernel<256, 6, 1, 1, 1, 1, 0>"
    fp = workloads.Problem("f", torch.zeros(1, 1), torch.zeros(1, 1), Bs=torch.zeros(1, 1))
    p = binding.gemm_query_plan(16, 28672, 4096, fp4=True, sm_count=148)
    assert bench.kernel_key(p, fp) == "skinny_gemm_kernel<16, 4, 1, 0>"


def test_traffic_is_reported_only_for_current_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(
        {"source_hash": "not-the-current-hash", "kernels": {"k@w": {"dram_bytes_per_launch": 5}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "current")
    assert bench.stored_traffic("k@w") is None
    (prof / "traffic.json").write_text(json.dumps(
        {"source_hash": "current", "kernels": {"k@w": {"dram_bytes_per_launch": 5}}}))
    assert bench.stored_traffic("k@w") == 5
    assert bench.stored_traffic("other@w") is None


def test_clock_summary_counts_reasons_between_samples(tmp_path):
    """A slowdown reason that no 20 ms sample caught still shows up through the
    driver's cumulative counters read at the ends of the timed region; samples
    outside the region are dropped."""
    c = bench.ClockSampler(0)
    c.out.close()
    rows = [("2026/01/01 00:00:00.000", 2070, "0x0000000000000000", "Not Active"),
            ("2026/01/01 00:00:01.000", 2070, "0x0000000000000000", "Not Active"),
            ("2026/01/01 00:00:01.020", 1700, "0x0000000000000000", "Not Active"),
            ("2026/01/01 00:00:01.040", 1700, "0x0000000000000004", "Active"),
            ("2026/01/01 00:00:09.000", 900, "0x0000000000000040", "Not Active")]
    with open(c.out.name, "w") as f:
        for ts, sm, mask, cap in rows:
            f.write(f"{ts}, 0, {sm}, 2070, 300.5, {mask}, Not Active, Not Active, "
                    f"Not Active, {cap}, 900.25\n")
    import datetime
    t = lambda s: datetime.datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    c.t_start, c.t_end = t("2026/01/01 00:00:00.990"), t("2026/01/01 00:00:01.050")
    c.c_start = {"sw_power_cap": 100, "sw_thermal_slowdown": 5, "hw_thermal_slowdown": 0,
                 "hw_power_brake_slowdown": 0}
    c.c_end = dict(c.c_start, sw_power_cap=30100)
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1700 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["active_reasons"] == ["sw_power_cap"]
    assert s["reason_us"]["sw_power_cap"] == 30000 and s["reason_us"]["sw_thermal_slowdown"] == 0
    assert s["power_instant_w_max"] == 900.25 and s["window_us"] == 60000
    # without counters (older drivers) the samples alone decide
    c2 = bench.ClockSampler(0)
    c2.out.close()
    with open(c2.out.name, "w") as f:
        f.write("2026/01/01 00:00:01.020, 0, 1700, 2070, 300.5, 0x0000000000000000, "
                "Not Active, Not Active, Not Active, Not Active\n")
    c2.t_start, c2.t_end, c2.c_start, c2.c_end = None, None, None, None
    s2 = c2.summary()
    assert s2["reasons"] == [] and s2["reason_us"] is None and s2["power_instant_w_max"] == 300.5
