"""CPU tests of bench.py's host logic: the roofline arithmetic, the multi-rank
timing reduction (2 gloo ranks), the reference arm's JSON line and the
clock-sample parsing."""
from __future__ import annotations

import io
import json
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
    assert bench.profiled_traffic("no_such_kernel") is None


class _W:
    def __init__(self, m, n, k):
        self.m, self.n, self.k = m, n, k


def test_roofline_of_the_headline_is_hbm_bound():
    works = [_W(32, 4096, 512), _W(32, 2880, 512)]
    r = bench.dominant_roofline(works, [[9e-6, 9e-6], [9e-6, 9e-6]], 152)
    hbm, _, _ = bench.load_peaks()
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["kernel"] == "gemm_kernel<32, fused>"
    per_launch = (bench.algorithmic_bytes(32, 4096, 512) + bench.algorithmic_bytes(32, 2880, 512)) / 2
    assert r["algorithmic_bytes_per_launch"] == int(per_launch)
    assert abs(r["achieved"] - per_launch / 9e-6 / 1e9) < 0.01
    assert abs(r["frac"] - r["achieved"] / hbm) < 1e-4


def test_roofline_of_the_large_gemm_picks_the_longer_floor():
    hbm, bf16, _ = bench.load_peaks()
    # m = 4096, k = 2048: 83 MB of algorithmic bytes outlast 120 GFLOP at
    # the peaks (the C write dominates), so the bound is HBM
    r = bench.dominant_roofline([_W(4096, 7168, 2048)], [[40e-6, 40e-6]], 152)
    assert r["bound"] == "hbm" and r["kernel"] == "gemm_pair_kernel"
    assert abs(r["achieved"] - bench.algorithmic_bytes(4096, 7168, 2048) / 40e-6 / 1e9) < 0.01
    # a long K makes the FP4 work the longer floor: the measured bf16 peak
    # times the nominal FP4 / bf16 ratio (13.5 / 2.25)
    r = bench.dominant_roofline([_W(4096, 7168, 16384)], [[100e-6, 100e-6]], 152)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["kernel"] == "gemm_pair_kernel"
    assert abs(r["peak"] - bf16 * 6) < 0.1
    assert abs(r["achieved"] - 2 * 4096 * 7168 * 16384 / 100e-6 / 1e12) < 0.1


@pytest.mark.parametrize("m,n,name", [(4, 2880, "gemm_kernel<16, fused>"), (32, 4096, "gemm_kernel<32, fused>"),
                                      (64, 7168, "gemm_kernel<64, image swap>"),
                                      (256, 3072, "gemm_kernel<128, image plain>"), (4096, 7168, "gemm_pair_kernel")])
def test_kernel_labels_follow_the_planner(m, n, name):
    assert bench.gemm_kernel_name(m, n, 152) == name
    assert bench.launches_per_gemm(m) == (1 if m <= 32 else 2)
