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
