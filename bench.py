"""Benchmark of the MXFP4 GEMM hot path  C = quant(A) . B^T  on GB300.

One step = one pass of the whole hot path over one batch of synthetic input
for the headline workload: the two m=32, k=512 shapes (n=4096 and n=2880) of
the "kernelbot amd-mxfp4-mm" leaderboard set, each a single fused launch
(A quantized in-kernel, block-scaled tcgen05 MMA, bf16 epilogue).  B is
quantized and prepacked once, untimed.  L2 is flushed (a write larger than
L2) before every timed GEMM; each GEMM is timed with CUDA events on its
launch stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME[,NAME]] [--table]

Prints one JSON line on rank 0.  --table also prints per-shape results for
every workload to stderr.  --impl reference times the CPU oracle instead
(the only other place besides cpu_baseline where this script runs it).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MXFP4 GEMM µs + effective TB/s per shape (L2-cold); % of HBM/FP4 roofline"
NOMINAL_FP4_TFLOPS = 13500.0  # dense FP4 tensor rate, nominal (no measured FP4 peak is available)
NOMINAL_BF16_TFLOPS = 2250.0  # dense bf16 tensor rate, nominal (for the FP4/bf16 ratio)


def algorithmic_bytes(m, n, k):
    """bf16 A + fp4 B + e8m0 B scales + bf16 C: what any implementation must move."""
    return 2 * m * k + n * k // 2 + n * k // 32 + 2 * m * n


def flops(m, n, k):
    return 2 * m * n * k


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# the files that compile into the kernels (the C-ABI glue in mxfp4_api.cu and
# mxfp4_noalloc.cu only validates arguments and calls the launchers)
KERNEL_SOURCES = ("mxfp4_device.cuh", "mxfp4_gemm.cu", "mxfp4_launch.h", "mxfp4_quant.cu", "ptx.cuh")


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "precision_bf16_mxfp4_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        entry = t[kernel_key]
        if entry.get("source_hash") == source_hash():
            return int(entry["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampler run around the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ ours
def run_ours(args, names, rank, world, local_rank):
    import numpy as np
    import torch

    import precision_bf16_mxfp4_gb300 as mx
    from precision_bf16_mxfp4_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    shapes = []
    for nm in names:
        w = inputs.WORKLOADS[nm]
        a, b = inputs.make_inputs(nm, seed=0)
        a_dev, b_dev = a.to(dev), b.to(dev)
        # B: quantized on the device by the library's own quantizer (bit-identical
        # to the oracle, checked by the GPU tests), prepacked once, untimed
        bq, bs = mx.quant(b_dev)
        packed = mx.prepack_b(bq, bs)
        del bq, bs, b_dev
        c = torch.empty((w.m, w.n), dtype=torch.bfloat16, device=dev)
        ws_bytes = mx.workspace_bytes(w.m, w.n, w.k)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
        a_host = a.pin_memory()
        c_host = torch.empty((w.m, w.n), dtype=torch.bfloat16).pin_memory()
        shapes.append(dict(w=w, a=a_dev, packed=packed, c=c, ws=ws, a_host=a_host, c_host=c_host))
    torch.cuda.synchronize()

    def step_device(evs):
        for i, s in enumerate(shapes):
            flush.zero_()
            evs[i][0].record(stream)
            mx.gemm(s["a"], s["packed"], out=s["c"], workspace=s["ws"])
            evs[i][1].record(stream)

    def step_e2e(evs):
        for i, s in enumerate(shapes):
            flush.zero_()
            evs[i][0].record(stream)
            # one C-ABI call with host buffers: A up, the GEMM, C down
            mx.gemm_host(s["a_host"], s["packed"], out=s["c_host"], a_dev=s["a"], c_dev=s["c"], workspace=s["ws"])
            evs[i][1].record(stream)

    def timed(step_fn, steps):
        evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in shapes] for _ in range(steps)]
        for _ in range(args.warmup):
            step_fn([[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in shapes])
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            step_fn(evs[k])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(world)
        per_shape = [[evs[k][i][0].elapsed_time(evs[k][i][1]) * 1e-3 for k in range(steps)] for i in range(len(shapes))]
        return per_shape, wall

    with ClockSampler(local_rank) as clk:
        dev_times, wall = timed(step_device, args.steps)
    e2e_times, _ = timed(step_e2e, max(args.steps // 4, 3))
    mx.device_status(dev)

    step_bytes = sum(algorithmic_bytes(s["w"].m, s["w"].n, s["w"].k) for s in shapes)
    step_s = sum(statistics.mean(t) for t in dev_times)
    step_s_max = max_over_ranks(step_s, world)
    e2e_s = max_over_ranks(sum(statistics.mean(t) for t in e2e_times), world)
    hbm_gbs, _, peak_src = load_peaks()

    shape_rows = []
    for s, t in zip(shapes, dev_times):
        w = s["w"]
        med = statistics.median(t)
        byt, fl = algorithmic_bytes(w.m, w.n, w.k), flops(w.m, w.n, w.k)
        floor_s = max(byt / (hbm_gbs * 1e9), fl / (NOMINAL_FP4_TFLOPS * 1e12))
        shape_rows.append({"shape": w.name, "m": w.m, "n": w.n, "k": w.k, "us_median": round(med * 1e6, 3),
                           "us_mean": round(statistics.mean(t) * 1e6, 3),
                           "tbps": round(byt / med / 1e12, 4), "tflops": round(fl / med / 1e12, 3),
                           "roofline_frac": round(floor_s / med, 4)})

    roofline = dominant_roofline([s["w"] for s in shapes], dev_times, props.multi_processor_count)

    out = {
        "metric": METRIC, "value": round(world * step_bytes / step_s_max / 1e12, 5), "unit": "TB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s_max * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in, e2m1 x e2m1 -> fp32 accumulate, bf16 out",
        "data": "synthetic (seeded N(0,1) A and B, B quantized on device and prepacked once)",
        "config": {"workload": "+".join(names), "shapes": [[s["w"].m, s["w"].n, s["w"].k] for s in shapes],
                   "l2": "flushed before every timed GEMM (write of %d MiB)" % (flush.numel() >> 20),
                   "parallelism": f"replicas x{world}"},
        "shapes": shape_rows,
        "e2e": {"value": round(world * step_bytes / e2e_s / 1e12, 5), "unit": "TB/s",
                "us_per_step": round(e2e_s * 1e6, 3),
                "h2d_bytes_per_step": int(sum(s["a_host"].numel() * 2 for s in shapes)),
                "d2h_bytes_per_step": int(sum(s["c_host"].numel() * 2 for s in shapes))},
        "gpu_launches": args.steps * sum(launches_per_gemm(s["w"].m) for s in shapes),
        "roofline": roofline,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
    }
    if args.table and rank == 0:
        print_table(dev, flush, mx, inputs, hbm_gbs)
    return out


def launches_per_gemm(m):
    """Kernels one mxfp4_gemm call launches: the fused GEMM alone for m <= 32,
    else the activation quantizer and the GEMM."""
    return 1 if m <= 32 else 2


def gemm_kernel_name(m, n, sms):
    """The GEMM kernel the library's planner picks for (m, n) (its rule,
    restated for labelling the roofline)."""
    if m <= 32:
        return "gemm_kernel<%d, fused>" % (16 if m <= 16 else 32)
    if m <= 128:
        return "gemm_kernel<%d, image swap>" % (64 if m <= 64 else 128)
    if n >= 256 and -(-m // 128) * -(-n // 256) >= sms:
        return "gemm_pair_kernel"
    return "gemm_kernel<128, image plain>"


def dominant_roofline(works, dev_times, sms):
    """Roofline of the step's dominant GEMM (the shape with the most FLOPs),
    bound by whichever floor is longer at the measured peaks.  HBM-bound
    (the m <= 32 headline, and m = 4096 with k = 2048): algorithmic bytes per
    launch over the mean event time per launch against the measured copy
    bandwidth.  A shape whose FP4 work
    outweighs its bytes at the peaks (a long-K large-m GEMM; m = 4096 with
    k = 2048 is still bound by its 56 MiB of C): algorithmic FLOPs over the
    mean event time of its step, which also covers the activation quantizer
    that precedes the GEMM (a lower bound for the GEMM alone), against the
    measured bf16 peak times NVIDIA's nominal FP4/bf16 ratio (13.5 / 2.25)."""
    hbm_gbs, bf16_tflops, peak_src = load_peaks()
    fp4_peak = bf16_tflops * (NOMINAL_FP4_TFLOPS / NOMINAL_BF16_TFLOPS)
    i = max(range(len(works)), key=lambda j: flops(works[j].m, works[j].n, works[j].k))
    w = works[i]
    fl, byt = flops(w.m, w.n, w.k), algorithmic_bytes(w.m, w.n, w.k)
    kernel = gemm_kernel_name(w.m, w.n, sms)
    if fl / (fp4_peak * 1e12) > byt / (hbm_gbs * 1e9):
        t = statistics.mean(dev_times[i])
        achieved = fl / t / 1e12
        return {"bound": "tensor", "kernel": kernel, "achieved": round(achieved, 1), "peak": round(fp4_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / fp4_peak, 4),
                "peak_source": f"{peak_src} bf16_tflops x nominal FP4/bf16 ratio 6",
                "traffic": profiled_traffic("gemm_pair_m4096") if (w.m, w.n, w.k) == (4096, 7168, 2048) else None,
                "algorithmic_flops_per_launch": int(fl),
                "timed": "event pair around quantizer + GEMM (one step of this shape)"}
    # bandwidth-bound: bytes per launch over the mean time per launch, all shapes
    kernel_s = sum(statistics.mean(t) for t in dev_times) / len(works)
    kernel_bytes = sum(algorithmic_bytes(x.m, x.n, x.k) for x in works) / len(works)
    achieved = kernel_bytes / kernel_s / 1e9
    if all(16 < x.m <= 32 for x in works):
        traffic = profiled_traffic("gemm_fused_bn32")
    elif [(x.m, x.n, x.k) for x in works] == [(4096, 7168, 2048)]:
        traffic = profiled_traffic("gemm_pair_m4096")
    else:
        traffic = None
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 2),
            "peak": hbm_gbs, "unit": "GB/s", "frac": round(achieved / hbm_gbs, 4),
            "peak_source": f"{peak_src} hbm_gbs", "traffic": traffic,
            "algorithmic_bytes_per_launch": int(kernel_bytes)}


def print_table(dev, flush, mx, inputs, hbm_gbs, table_iters=200):
    import torch
    stream = torch.cuda.current_stream(dev)
    print(f"{'workload':22s} {'us mean':>9s} {'median':>8s} {'TB/s':>7s} {'TFLOP/s':>8s} {'roof':>6s}", file=sys.stderr)
    for nm, w in inputs.WORKLOADS.items():
        a, b = inputs.make_inputs(nm, seed=0)
        a_dev = a.to(dev)
        bq, bs = mx.quant(b.to(dev))
        packed = mx.prepack_b(bq, bs)
        c = torch.empty((w.m, w.n), dtype=torch.bfloat16, device=dev)
        wsb = mx.workspace_bytes(w.m, w.n, w.k)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev) if wsb else None
        ts = []
        for it in range(5 + table_iters):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            mx.gemm(a_dev, packed, out=c, workspace=ws)
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= 5:
                ts.append(e0.elapsed_time(e1) * 1e-3)
        # the event clock ticks in steps of about 1 us: the mean over many
        # launches resolves finer than any single sample or the median
        mean, med = statistics.mean(ts), statistics.median(ts)
        byt, fl = algorithmic_bytes(w.m, w.n, w.k), flops(w.m, w.n, w.k)
        floor_s = max(byt / (hbm_gbs * 1e9), fl / (NOMINAL_FP4_TFLOPS * 1e12))
        print(f"{nm:22s} {mean*1e6:9.2f} {med*1e6:8.2f} {byt/mean/1e12:7.3f} {fl/mean/1e12:8.1f} {floor_s/mean:6.3f}",
              file=sys.stderr)


# ------------------------------------------------------------ CPU oracle
def _oracle_prepare(names, fraction):
    """Inputs for the oracle step: each shape's A and the first `fraction` of
    its weight rows (output columns), B quantized by the oracle."""
    import oracle
    from precision_bf16_mxfp4_gb300 import inputs
    prepared = []
    for nm in names:
        w = inputs.WORKLOADS[nm]
        a, b = inputs.make_inputs(nm, seed=0)
        ns = max(1, int(round(w.n * fraction)))
        bits = lambda t: t.contiguous().view(__import__("torch").int16).numpy().view("uint16")
        bq, bs = oracle.quant(bits(b[:ns]))
        prepared.append((w, bits(a), bq, bs, ns))
    return prepared


def _oracle_run(prepared):
    """The oracle (quant of A, then the fp64 GEMM) on prepared inputs.
    Returns (seconds, algorithmic bytes covered)."""
    import oracle
    t0 = time.perf_counter()
    covered = 0
    for w, a_bits, bq, bs, ns in prepared:
        aq, a_s = oracle.quant(a_bits)
        oracle.gemm(aq, a_s, bq, bs)
        covered += algorithmic_bytes(w.m, ns, w.k)
    return time.perf_counter() - t0, covered


def oracle_step_sample(names, fraction):
    """The oracle on the first `fraction` of each shape's output columns."""
    return _oracle_run(_oracle_prepare(names, fraction))


def cpu_baseline(names, budget_s=12.0):
    """The oracle on 1/8 of each shape's output columns, repeated until about
    `budget_s` seconds of single-threaded CPU work have been timed."""
    prepared = _oracle_prepare(names, 0.125)
    total_t, total_b, reps = 0.0, 0, 0
    while total_t < budget_s and reps < 10000:
        dt, cb = _oracle_run(prepared)
        total_t += dt
        total_b += cb
        reps += 1
    return {"value": round(total_b / total_t / 1e12, 9), "unit": "TB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} x (quant of A + fp64 GEMM on 1/8 of each shape's output columns), "
                      f"single-threaded C, {total_t:.1f} s"}


def run_reference(args, names):
    # size the per-step sample so that warmup + steps end within about a minute
    t_probe, b_probe = oracle_step_sample(names, 1.0 / 64)
    per_step_budget = 60.0 / max(1, args.steps + args.warmup)
    frac = max(1.0 / 4096, min(1.0, per_step_budget / max(t_probe, 1e-4) / 64))
    for _ in range(args.warmup):
        oracle_step_sample(names, frac)
    times, covered = [], 0
    for _ in range(args.steps):
        dt, cb = oracle_step_sample(names, frac)
        times.append(dt)
        covered = cb
    step_s = statistics.mean(times)
    value = covered / step_s / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 9), "unit": "TB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": "+".join(names), "sample_fraction_of_columns": frac},
        "cpu_baseline": {"value": round(value, 9), "unit": "TB/s", "cores": 1, "kind": "oracle",
                         "sample": f"quant of A + fp64 GEMM on {frac:.5f} of each shape's output columns per step"},
        "e2e": {"value": round(value, 9), "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------ distributed
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measure_fp4_peak(local_rank, kblocks_per_sm=4000, runs=5):
    """The dense FP4 tensor-core rate (the large-m GEMM's roofline
    denominator, which the measured-peaks file does not provide): the
    median of `runs` launches of the library's microbenchmark, with the SM
    clocks sampled meanwhile."""
    import torch

    import precision_bf16_mxfp4_gb300 as mx
    torch.cuda.set_device(local_rank)
    mx.measure_fp4_peak(200)  # warm-up: module load, attributes
    with ClockSampler(local_rank) as clk:
        vals = [mx.measure_fp4_peak(kblocks_per_sm) for _ in range(runs)]
    return {"fp4_peak_tflops": round(statistics.median(vals), 1), "runs_tflops": [round(v, 1) for v in vals],
            "kblocks_per_sm": kblocks_per_sm, "sms": torch.cuda.get_device_properties(local_rank).multi_processor_count,
            "nominal_tflops": NOMINAL_FP4_TFLOPS, "clocks": clk.summary()}


def measure_launch_floor(local_rank, steps, warmup, ctas=32):
    """The launch floor of the small-m GEMMs: CUDA events around one empty
    kernel, and around two back to back, each after the same L2 flush the
    GEMMs get (mean and median over `steps`, in microseconds)."""
    import torch

    import precision_bf16_mxfp4_gb300 as mx
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    out = {"ctas": ctas, "steps": steps, "l2": "flushed before every timed launch (write of %d MiB)" %
           (flush.numel() >> 20)}
    for count in (1, 2):
        times = []
        for it in range(warmup + steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mx.launch_empty(count, ctas)
            e1.record()
            torch.cuda.synchronize()
            if it >= warmup:
                times.append(e0.elapsed_time(e1) * 1e3)
        out[f"{count}_kernel_us"] = {"mean": round(statistics.mean(times), 3), "median": round(statistics.median(times), 3)}
    return out


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="m32_n4096_k512,m32_n2880_k512")
    p.add_argument("--table", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--fp4-peak", action="store_true",
                   help="measure the dense FP4 tensor-core rate (mxfp4_measure_fp4_peak) and exit")
    p.add_argument("--launch-floor", action="store_true",
                   help="time one and two empty kernels with the GEMMs' flush + event method and exit")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    names = args.workload.split(",")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, names)))
        return 0

    if args.fp4_peak:
        if rank == 0:
            print(json.dumps(measure_fp4_peak(local_rank)))
        return 0

    if args.launch_floor:
        if rank == 0:
            print(json.dumps(measure_launch_floor(local_rank, args.steps, args.warmup)))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    out = run_ours(args, names, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(names)
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
