"""CPU tests of bench.py's host logic: the roofline arithmetic, the multi-rank
timing reduction (2 gloo ranks), the reference arm's JSON line and the
clock-sample parsing."""
from __future__ import annotations

import io
import json
import os
import socket
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

import bench
from tests.helpers import gloo_max_over_ranks_worker

# 2mk + nk/2 + nk/32 + 2mn for the seven workloads, computed by hand
EXPECTED_BYTES = {
    (4, 2880, 512): 810_496,
    (32, 4096, 512): 1_409_024,
    (32, 2880, 512): 1_000_448,
    (16, 2112, 7168): 8_339_456,
    (64, 7168, 2048): 8_978_432,
    (256, 3072, 1536): 4_866_048,
    (4096, 7168, 2048): 83_296_256,
}


@pytest.mark.parametrize("shape", list(EXPECTED_BYTES))
def test_algorithmic_bytes(shape):
    assert bench.algorithmic_bytes(*shape) == EXPECTED_BYTES[shape]
    m, n, k = shape
    assert bench.flops(m, n, k) == 2 * m * n * k


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    values = [0.25, 1.5]
    port = _free_port()
    procs = [ctx.Process(target=gloo_max_over_ranks_worker, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 1.5, 1: 1.5}


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.0, 1) == 3.0


def test_reference_arm_json_line(monkeypatch):
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3", "--workload", "m4_n2880_k512"]) == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TB/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["host_cores"] >= 1 and line["cpu_baseline"]["cpu_model"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert buf.getvalue() == ""


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_clock_summary_flags_throttle_reasons():
    c = bench.ClockSampler(0)
    c.lines = ["2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
               "1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
               "2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    c.lines = []
    assert c.summary()["reasons"] == ["unsampled"]


def test_traffic_is_reported_only_for_the_profiled_sources():
    assert bench.profiled_traffic("no_such_shape") is None
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for name, entry in t["shapes"].items():
        m = int(name.split("_")[0][1:])
        kernels = entry["kernels"]
        assert len(kernels) == bench.launches_per_gemm(m), name
        total = sum(v["dram_read"] + v["dram_write"] for v in kernels.values())
        got = bench.profiled_traffic(name, bench.launches_per_gemm(m))
        # the captured figure, or nothing once the kernel sources have changed
        assert got == (total if t["source_hash"] == bench.source_hash() else None)
        # a call with another number of kernels is never given this capture
        assert bench.profiled_traffic(name, bench.launches_per_gemm(m) + 1) is None


class _W:
    def __init__(self, m, n, k, name="w"):
        self.m, self.n, self.k, self.name = m, n, k, name


def test_fp4_peak_is_the_measured_bf16_rate_times_six():
    _, bf16, _ = bench.load_peaks()
    fp4, _ = bench.fp4_peak_tflops()
    assert abs(fp4 - bf16 * 6.0) < 1e-6


def test_every_benchmark_shape_is_hbm_bound_at_the_peaks():
    # the algorithmic bytes at the HBM peak outlast the FLOPs at the FP4 peak
    # for all seven shapes (m=4096: 83 MB vs 120 GFLOP, the C write dominates)
    for shape in EXPECTED_BYTES:
        t, bound = bench.shape_floor(*shape)
        hbm, _, _ = bench.load_peaks()
        assert bound == "hbm" and abs(t - EXPECTED_BYTES[shape] / (hbm * 1e9)) < 1e-12


def test_shape_row_fraction_and_launch_floor_multiple():
    w = _W(32, 4096, 512, "m32_n4096_k512")
    row = bench.shape_row(w, [9e-6, 10e-6, 11e-6], {1: 5.0, 2: 7.0}, 152)
    hbm, _, _ = bench.load_peaks()
    assert row["us_mean"] == 10.0 and row["us_median"] == 10.0 and row["us_trimmed"] == 10.0
    assert bench.trimmed_mean([1.0, 5.0, 6.0, 7.0, 100.0]) == 6.0
    assert abs(row["frac"] - EXPECTED_BYTES[(32, 4096, 512)] / (hbm * 1e9) / 10e-6) < 1e-4
    assert row["launches"] == 1 and row["launch_floor_us"] == 5.0 and row["x_launch_floor"] == 2.0
    row2 = bench.shape_row(_W(64, 7168, 2048, "m64"), [14e-6], {1: 5.0, 2: 7.0}, 152)
    assert row2["launches"] == 2 and row2["launch_floor_us"] == 7.0 and row2["x_launch_floor"] == 2.0
    assert row2["kernels"] == "quant_image_kernel + gemm_kernel<64, image swap>"
    assert "x_minimal_floor" not in row2
    floors = {1: 5.0, 2: 7.0, ("minimal", 1): 6.0, ("minimal", 2): 8.0}
    row3 = bench.shape_row(w, [12e-6], floors, 152)
    assert row3["minimal_floor_us"] == 6.0 and row3["x_minimal_floor"] == 2.0 and row3["x_launch_floor"] == 2.4
    row4 = bench.shape_row(_W(64, 7168, 2048, "m64"), [12e-6], floors, 152)
    assert row4["minimal_floor_us"] == 8.0 and row4["x_minimal_floor"] == 1.5


def test_roofline_picks_the_slowest_call_and_its_floor():
    hbm, bf16, _ = bench.load_peaks()
    works = [_W(32, 4096, 512, "a"), _W(4096, 7168, 2048, "b")]
    r = bench.dominant_roofline(works, [[9e-6, 9e-6], [40e-6, 40e-6]], 152)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["shape"] == "b"
    assert r["kernel"] == "quant_image_kernel + gemm_pair_kernel"
    assert r["algorithmic_bytes_per_launch"] == EXPECTED_BYTES[(4096, 7168, 2048)]
    assert abs(r["achieved"] - EXPECTED_BYTES[(4096, 7168, 2048)] / 40e-6 / 1e9) < 0.01
    assert abs(r["frac"] - r["achieved"] / hbm) < 1e-4
    # a long K makes the FP4 work the longer floor: the measured bf16 peak
    # times the nominal FP4 / bf16 ratio (13.5 / 2.25)
    r = bench.dominant_roofline([_W(4096, 7168, 16384, "c")], [[100e-6, 100e-6]], 152)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["peak"] - bf16 * 6) < 0.1
    assert abs(r["achieved"] - 2 * 4096 * 7168 * 16384 / 100e-6 / 1e12) < 0.1


def test_oracle_sample_is_bounded():
    assert bench.sample_of(_W(4096, 7168, 2048)) == (256, 896)
    assert bench.sample_of(_W(16, 2112, 7168)) == (16, 264)
    assert bench.sample_of(_W(4, 2880, 512)) == (4, 360)


def test_default_workload_is_the_seven_shapes():
    from precision_bf16_mxfp4_gb300 import inputs
    names = bench.DEFAULT_WORKLOAD.split(",")
    assert len(names) == 7 and set(names) == set(inputs.WORKLOADS)
    assert {(inputs.WORKLOADS[n].m, inputs.WORKLOADS[n].n, inputs.WORKLOADS[n].k) for n in names} == set(EXPECTED_BYTES)


def test_host_cpu_reports_cores_and_a_model():
    cores, model = bench.host_cpu()
    assert cores >= 1 and isinstance(model, str) and model


@pytest.mark.parametrize("m,n,name", [(4, 2880, "gemm_kernel<16, fused>"), (32, 4096, "gemm_kernel<32, fused>"),
                                      (64, 7168, "gemm_kernel<64, image swap>"),
                                      (256, 3072, "gemm_kernel<128, image plain>"), (4096, 7168, "gemm_pair_kernel")])
def test_kernel_labels_follow_the_planner(m, n, name):
    assert bench.gemm_kernel_name(m, n, 152) == name
    assert bench.launches_per_gemm(m) == (1 if m <= 32 else 2)
