"""Host-side logic of bench.py that needs no GPU: the whole-job aggregation over
ranks (two gloo processes on the CPU), kernel naming and the traffic lookup."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from tensor_core_gemm_02_gb300 import binding, workloads  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [2.0, 3.0][rank]  # rank 1 is the slow one
    ms = bench.slowest_rank(local_ms, world, torch.device("cpu"))
    value = bench.job_throughput(1e12, ms, world)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        ms, value = res[rank]
        assert ms == 3.0
        # 2 ranks x 1 TFLOP each over 3 ms
        assert abs(value - 2 * 1e12 / 3e-3 / 1e12) < 1e-9


def test_single_rank_needs_no_process_group():
    assert bench.slowest_rank(1.5, 1, torch.device("cpu")) == 1.5
    assert bench.job_throughput(2e12, 2.0, 1) == pytest.approx(1000.0)


def test_kernel_keys_name_the_launched_instance():
    binding.load_library()
    p = binding.gemm_query_plan(8192, 8192, 8192, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 1, 2, 1, 0>"
    p = binding.gemm_query_plan(8192, 28672, 4096, has_c=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 6, 1, 1, 1, 0>"
    p = binding.gemm_query_plan(16, 28672, 4096, sm_count=148)
    assert bench.kernel_key(p) == "skinny_gemm_kernel<16, 1, 0>"
    p = binding.gemm_query_plan(1024, 1024, 1024, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<64, 8, 0, 1, 1, 0>"
    p = binding.gemm_query_plan(16384, 4096, 4096, gather=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 1, 2, 4, 0>"
    p = binding.gemm_query_plan(16384, 1024, 4096, gather=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 1, 2, 2, 0>"
    p = binding.gemm_query_plan(16384, 1024, 1024, gather=True, sm_count=148)
    assert bench.kernel_key(p) == "tile_gemm_kernel<256, 4, 0, 1, 4, 0>"
    # the epilogue mode and the FP4 converter warps come from the problem
    sc = workloads.Problem("s", torch.zeros(1, 1), torch.zeros(1, 1), idx=torch.zeros(1),
                           scatter=True, d_rows=1)
    p = binding.gemm_query_plan(16384, 4096, 4096, scatter=True, sm_count=148)
    assert bench.kernel_key(p, sc) == "tile_gemm_kernel<256, 6, 1, 1, 1, 1>"
    fp = workloads.Problem("f", torch.zeros(1, 1), torch.zeros(1, 1), Bs=torch.zeros(1, 1))
    p = binding.gemm_query_plan(16, 28672, 4096, fp4=True, sm_count=148)
    assert bench.kernel_key(p, fp) == "skinny_gemm_kernel<16, 4, 1>"


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
