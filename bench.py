"""Benchmark of the MXFP4 GEMM hot path  C = quant(A) . B^T  on GB300.

One step = one pass of the whole hot path over the seven shapes of the
"kernelbot amd-mxfp4-mm" benchmark set (submission 752099, module docstring
shape list, plus the compute-heavy m=4096 case):

    m4_n2880_k512, m32_n4096_k512, m32_n2880_k512, m16_n2112_k7168,
    m64_n7168_k2048, m256_n3072_k1536, m4096_n7168_k2048

each one mxfp4_gemm call (bf16 A quantized on the fly, block-scaled tcgen05
MMA, bf16 C).  B is quantized and prepacked once, untimed.  L2 is flushed (a
write larger than L2) before every timed GEMM and each GEMM is timed with
CUDA events on its launch stream.  `value` = algorithmic bytes of the step /
summed event time (TB/s); `shapes` has one row per shape (us, TB/s, TFLOP/s,
roofline fraction and bound, launch-floor multiple, parity).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME[,NAME]] [--no-cpu-baseline]
                    [--fp4-peak | --launch-floor]

Prints one JSON line on rank 0.  The CPU oracle runs in two places only: the
cpu_baseline leg (rank 0 at N=1, before timing: it also checks the GPU's
output on its sample, the in-process parity check) and --impl reference.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MXFP4 GEMM µs + effective TB/s per shape (L2-cold); % of HBM/FP4 roofline"
NOMINAL_FP4_TFLOPS = 13500.0  # NVIDIA's dense FP4 figure for GB300 (context only)
NOMINAL_BF16_TFLOPS = 2250.0  # NVIDIA's dense bf16 figure (for the FP4/bf16 ratio)
DEFAULT_WORKLOAD = ("m4_n2880_k512,m32_n4096_k512,m32_n2880_k512,m16_n2112_k7168,"
                    "m64_n7168_k2048,m256_n3072_k1536,m4096_n7168_k2048")
# |gpu - ref| <= 2^-7 |ref| + 1e-3 max|ref| (exact e2m1 products; only the fp32
# summation order and the final bf16 rounding differ from the fp64 oracle)
REL_TOL, ABS_TOL_FRAC = 2.0 ** -7, 1e-3


def algorithmic_bytes(m, n, k):
    """bf16 A + fp4 B + e8m0 B scales + bf16 C: what any implementation must move."""
    return 2 * m * k + n * k // 2 + n * k // 32 + 2 * m * n


def flops(m, n, k):
    return 2 * m * n * k


def load_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source) from the measured-peaks file."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def fp4_peak_tflops():
    """The FP4 roofline denominator used for every fraction: the measured
    dense bf16 rate times NVIDIA's nominal FP4/bf16 ratio (13.5 / 2.25)."""
    _, bf16, src = load_peaks()
    return bf16 * (NOMINAL_FP4_TFLOPS / NOMINAL_BF16_TFLOPS), src


def shape_floor(m, n, k):
    """(seconds, bound) of the roofline floor of one GEMM: the longer of its
    algorithmic bytes at the HBM peak and its FLOPs at the FP4 peak."""
    hbm_gbs, _, _ = load_peaks()
    fp4, _ = fp4_peak_tflops()
    t_mem = algorithmic_bytes(m, n, k) / (hbm_gbs * 1e9)
    t_fp4 = flops(m, n, k) / (fp4 * 1e12)
    return (t_mem, "hbm") if t_mem >= t_fp4 else (t_fp4, "tensor")


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


def profiled_traffic(shape_name, launches=None):
    """DRAM bytes (read + write) of one call on `shape_name`, summed over the
    call's kernels from the committed ncu captures, if they were taken on the
    current kernel sources and cover every kernel of the call; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("source_hash") != source_hash():
            return None
        kernels = t["shapes"][shape_name]["kernels"]
        if launches is not None and len(kernels) != launches:
            return None
        return int(sum(v["dram_read"] + v["dram_write"] for v in kernels.values()))
    except Exception:
        return None


def host_cpu():
    """(logical cores, CPU model) of this host."""
    model = platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip() + f" ({platform.machine()})"
                break
    except Exception:
        pass
    return os.cpu_count() or 1, model


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


def launches_per_gemm(m):
    """Kernels one mxfp4_gemm call launches: the fused GEMM alone for m <= 32,
    else the activation quantizer and the GEMM."""
    return 1 if m <= 32 else 2


def gemm_kernel_name(m, n, sms):
    """The GEMM kernel the library's planner picks for (m, n) (its rule,
    restated for labelling)."""
    if m <= 32:
        return "gemm_kernel<%d, fused>" % (16 if m <= 16 else 32)
    if m <= 128:
        return "gemm_kernel<%d, image swap>" % (64 if m <= 64 else 128)
    if n >= 256 and -(-m // 128) * -(-n // 256) >= sms:
        return "gemm_pair_kernel"
    return "gemm_kernel<128, image plain>"


def call_kernels(m, n, sms):
    """The kernels of one mxfp4_gemm call, in launch order."""
    g = gemm_kernel_name(m, n, sms)
    return g if m <= 32 else "quant_image_kernel + " + g


def trimmed_mean(times):
    """Mean without the single fastest and slowest time: the L2-cold timing
    of kernelbot amd-mxfp4-mm submission 739530 (its autotuning timer, which
    sorts the event times of a few runs and averages all but the two ends)."""
    ts = sorted(times)
    return statistics.mean(ts[1:-1]) if len(ts) > 2 else statistics.mean(ts)


def shape_row(w, times_s, floors_us, sms):
    """One per-shape result row from the event times (seconds) of its GEMMs."""
    mean, med = statistics.mean(times_s), statistics.median(times_s)
    byt, fl = algorithmic_bytes(w.m, w.n, w.k), flops(w.m, w.n, w.k)
    floor_s, bound = shape_floor(w.m, w.n, w.k)
    row = {"shape": w.name, "m": w.m, "n": w.n, "k": w.k, "kernels": call_kernels(w.m, w.n, sms),
           "launches": launches_per_gemm(w.m),
           "us_mean": round(mean * 1e6, 3), "us_median": round(med * 1e6, 3),
           "us_trimmed": round(trimmed_mean(times_s) * 1e6, 3),
           "tbps": round(byt / mean / 1e12, 4), "tflops": round(fl / mean / 1e12, 3),
           "bound": bound, "floor_us": round(floor_s * 1e6, 3), "frac": round(floor_s / mean, 4),
           "algorithmic_bytes": int(byt), "traffic": profiled_traffic(w.name, launches_per_gemm(w.m))}
    if floors_us:
        lf = floors_us.get(launches_per_gemm(w.m))
        if lf:
            row["launch_floor_us"] = lf
            row["x_launch_floor"] = round(mean * 1e6 / lf, 3)
        mf = floors_us.get(("minimal", launches_per_gemm(w.m)))
        if mf:
            row["minimal_floor_us"] = mf
            row["x_minimal_floor"] = round(mean * 1e6 / mf, 3)
    return row


def dominant_roofline(works, dev_times, sms, extra=None):
    """Roofline of the step's dominant call: the shape with the largest mean
    event time.  achieved = its algorithmic bytes (or FLOPs, if its FP4 work
    is the longer floor) per launch of the call / the call's mean event time,
    against the measured HBM copy bandwidth (or the FP4 peak of
    fp4_peak_tflops).  For m > 32 the call is two launches (the activation
    quantizer, then the GEMM as its programmatic dependent), timed together:
    an event between them would serialise what the dependent launch overlaps;
    `extra` carries the GEMM and the quantizer timed alone."""
    hbm_gbs, _, peak_src = load_peaks()
    fp4, fp4_src = fp4_peak_tflops()
    i = max(range(len(works)), key=lambda j: statistics.mean(dev_times[j]))
    w = works[i]
    t = statistics.mean(dev_times[i])
    fl, byt = flops(w.m, w.n, w.k), algorithmic_bytes(w.m, w.n, w.k)
    _, bound = shape_floor(w.m, w.n, w.k)
    kernel = call_kernels(w.m, w.n, sms)
    traffic = profiled_traffic(w.name, launches_per_gemm(w.m))
    out = {"bound": bound, "kernel": kernel, "shape": w.name,
           "traffic": traffic, "timed": "CUDA events around the whole call on its stream, mean over the timed steps"}
    if bound == "tensor":
        achieved = fl / t / 1e12
        out.update({"achieved": round(achieved, 1), "peak": round(fp4, 1), "unit": "TFLOP/s",
                    "frac": round(achieved / fp4, 4), "peak_source": f"{fp4_src} bf16_tflops x nominal FP4/bf16 6",
                    "algorithmic_flops_per_launch": int(fl)})
    else:
        achieved = byt / t / 1e9
        out.update({"achieved": round(achieved, 2), "peak": hbm_gbs, "unit": "GB/s",
                    "frac": round(achieved / hbm_gbs, 4), "peak_source": f"{peak_src} hbm_gbs",
                    "algorithmic_bytes_per_launch": int(byt)})
    if extra:
        out.update(extra)
    return out


# ------------------------------------------------------------------ ours
def make_flush(dev):
    import torch
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    return torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)


def event_time(stream, flush, fn, reps, warmup=3):
    """Mean and median seconds of fn() between CUDA events on `stream`, each
    repetition after an L2 flush."""
    import torch
    evs = []
    for r in range(warmup + reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        if r >= warmup:
            evs.append((e0, e1))
    torch.cuda.synchronize()
    t = [a.elapsed_time(b) * 1e-3 for a, b in evs]
    return statistics.mean(t), statistics.median(t)


def measure_launch_floor_live(dev, stream, flush, mx, reps):
    """Event time (us) of one and of two empty kernels after the same flush,
    and of one and two minimal kernels (a global read, a tensor-memory
    allocation and a global write per CTA: the least a GEMM launch does)."""
    out = {}
    for count in (1, 2):
        mean, med = event_time(stream, flush, lambda: mx.launch_empty(count, 32, dev), reps)
        out[count] = (round(mean * 1e6, 3), round(med * 1e6, 3))
        mean, med = event_time(stream, flush, lambda: mx.launch_minimal(count, 32, dev), reps)
        out[("minimal", count)] = (round(mean * 1e6, 3), round(med * 1e6, 3))
    return out


def run_ours(args, names, rank, world, local_rank):
    import numpy as np
    import torch

    import precision_bf16_mxfp4_gb300 as mx
    from precision_bf16_mxfp4_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    flush = make_flush(dev)

    shapes = []
    for nm in names:
        w = inputs.WORKLOADS[nm]
        a, b = inputs.make_inputs(nm, seed=0)
        a_dev, b_dev = a.to(dev), b.to(dev)
        # B: quantized on the device by the library's quantizer and prepacked
        # once, untimed; the cpu_baseline leg checks the quantized bytes
        # against the oracle's on its sample rows
        bq, bs = mx.quant(b_dev)
        packed = mx.prepack_b(bq, bs)
        ns = max(1, w.n // 8)
        bq_s, bs_s = bq[:ns].cpu().numpy(), bs[:ns].cpu().numpy()
        del bq, bs, b_dev
        c = torch.empty((w.m, w.n), dtype=torch.bfloat16, device=dev)
        ws_bytes = mx.workspace_bytes(w.m, w.n, w.k)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
        a_host = a.pin_memory()
        c_host = torch.empty((w.m, w.n), dtype=torch.bfloat16).pin_memory()
        shapes.append(dict(w=w, a_cpu=a, b_cpu=b, a=a_dev, packed=packed, c=c, ws=ws, a_host=a_host,
                           c_host=c_host, bq_s=bq_s, bs_s=bs_s))
    torch.cuda.synchronize()

    # one GEMM per shape for the parity check, run before anything is timed
    for s in shapes:
        mx.gemm(s["a"], s["packed"], out=s["c"], workspace=s["ws"])
    mx.device_status(dev)
    for s in shapes:
        s["c_first"] = s["c"].float().cpu().numpy()

    baseline, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        baseline, parity = cpu_baseline(shapes)

    reps = max(args.steps, 3)
    floors = measure_launch_floor_live(dev, stream, flush, mx, reps)
    fp4_measured = [mx.measure_fp4_peak(2000, dev) for _ in range(3)]

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
    # the last timed output still matches the first (checked) one bit for bit
    repeat_ok = all(np.array_equal(s["c"].float().cpu().numpy(), s["c_first"]) for s in shapes)
    host_us = host_call_overhead(mx, shapes, stream)

    # the dominant call's two kernels timed alone (outside the step), for the
    # roofline's split: the GEMM on a ready activation image, and the
    # activation quantizer
    works = [s["w"] for s in shapes]
    i_dom = max(range(len(shapes)), key=lambda j: statistics.mean(dev_times[j]))
    extra = None
    sd = shapes[i_dom]
    if sd["w"].m > 32:
        img = mx.quant_image(sd["a"])
        g_mean, g_med = event_time(stream, flush, lambda: mx.gemm_image(img, sd["packed"], out=sd["c"]), reps)
        q_mean, q_med = event_time(stream, flush, lambda: mx.quant_image(sd["a"], out=img), reps)
        hbm_gbs, _, _ = load_peaks()
        wd = sd["w"]
        gemm_bytes = wd.n * wd.k // 2 + wd.n * wd.k // 32 + 2 * wd.m * wd.n + mx.mxfp4_act_image_bytes(wd.m, wd.k)
        extra = {"gemm_alone": {"kernel": gemm_kernel_name(wd.m, wd.n, sms), "us_mean": round(g_mean * 1e6, 3),
                                "us_median": round(g_med * 1e6, 3),
                                "achieved_gbs": round(algorithmic_bytes(wd.m, wd.n, wd.k) / g_mean / 1e9, 1),
                                "frac": round(algorithmic_bytes(wd.m, wd.n, wd.k) / g_mean / 1e9 / hbm_gbs, 4),
                                "note": "mxfp4_gemm_image on a ready activation image (the call's algorithmic bytes "
                                        "over the GEMM's own time; its own operand bytes are %d)" % gemm_bytes},
                 "quantizer_alone": {"kernel": "quant_image_kernel", "us_mean": round(q_mean * 1e6, 3),
                                     "us_median": round(q_med * 1e6, 3),
                                     "bytes": 2 * wd.m * wd.k + mx.mxfp4_act_image_bytes(wd.m, wd.k)}}
        del img

    step_bytes = sum(algorithmic_bytes(s["w"].m, s["w"].n, s["w"].k) for s in shapes)
    step_s = sum(statistics.mean(t) for t in dev_times)
    step_s_max = max_over_ranks(step_s, world)
    e2e_s = max_over_ranks(sum(statistics.mean(t) for t in e2e_times), world)
    hbm_gbs, bf16, peak_src = load_peaks()
    fp4, fp4_src = fp4_peak_tflops()

    floors_mean = {c: v[0] for c, v in floors.items()}
    shape_rows = [shape_row(s["w"], t, floors_mean, sms) for s, t in zip(shapes, dev_times)]
    for r, s in zip(shape_rows, shapes):
        r["parity"] = parity[s["w"].name] if parity else "not checked (--no-cpu-baseline or N > 1)"
    roofline = dominant_roofline(works, dev_times, sms, extra)

    out = {
        "metric": METRIC, "value": round(world * step_bytes / step_s_max / 1e12, 5), "unit": "TB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s_max * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in, e2m1 x e2m1 -> fp32 accumulate, bf16 out",
        "data": "synthetic (seeded A and B per shape recipe; B quantized on device and prepacked once)",
        "config": {"workload": "+".join(names), "shapes": [[s["w"].m, s["w"].n, s["w"].k] for s in shapes],
                   "l2": "flushed before every timed GEMM (write of %d MiB)" % (flush.numel() >> 20),
                   "parallelism": f"replicas x{world}"},
        "shapes": shape_rows,
        "peaks": {"hbm_gbs": hbm_gbs, "hbm_source": peak_src, "fp4_tflops": round(fp4, 1),
                  "fp4_source": f"{fp4_src} bf16_tflops {bf16} x nominal FP4/bf16 ratio 6",
                  "fp4_peak_measured_tflops": round(statistics.median(fp4_measured), 1),
                  "fp4_peak_measured_note": "mxfp4_measure_fp4_peak: dense tcgen05 kind::mxf4, one CTA per SM, "
                                            "median of 3 launches",
                  "fp4_nominal_tflops": NOMINAL_FP4_TFLOPS},
        "launch_floor": {"1_kernel_us": {"mean": floors[1][0], "median": floors[1][1]},
                         "2_kernel_us": {"mean": floors[2][0], "median": floors[2][1]},
                         "1_minimal_kernel_us": {"mean": floors[("minimal", 1)][0],
                                                 "median": floors[("minimal", 1)][1]},
                         "2_minimal_kernel_us": {"mean": floors[("minimal", 2)][0],
                                                 "median": floors[("minimal", 2)][1]},
                         "method": "mxfp4_launch_empty (32 empty CTAs) and mxfp4_launch_minimal (32 CTAs that "
                                   "each read a word, allocate and free tensor memory and write a word) between "
                                   f"the same events after the same flush, {reps} repetitions; shapes carry "
                                   "x_launch_floor (empty) and x_minimal_floor"},
        "e2e": {"value": round(world * step_bytes / e2e_s / 1e12, 5), "unit": "TB/s",
                "us_per_step": round(e2e_s * 1e6, 3),
                "h2d_bytes_per_step": int(sum(s["a_host"].numel() * 2 for s in shapes)),
                "d2h_bytes_per_step": int(sum(s["c_host"].numel() * 2 for s in shapes)),
                "api": "mxfp4_gemm_host per shape (page-locked host A and C)"},
        "gpu_launches": args.steps * sum(launches_per_gemm(s["w"].m) for s in shapes),
        "roofline": roofline,
        "clocks": clk.summary(),
        "repeat_bit_identical": repeat_ok,
        "host_us_per_call": host_us,
        "wall_s_timed_region": round(wall, 4),
    }
    if baseline:
        out["cpu_baseline"] = baseline
    return out


def host_call_overhead(mx, shapes, stream, calls=200):
    """Host time per mxfp4_gemm call through the raw C ABI (arguments
    prebuilt, no synchronization inside the loop: the enqueue cost a caller
    pays), per shape, in microseconds; the ctypes call itself is included."""
    import ctypes
    import torch
    lib = mx._lib.load()
    P = ctypes.c_void_p
    out = {}
    for s in shapes:
        w = s["w"]
        ws = s["ws"]
        argv = (P(s["a"].data_ptr()), w.m, w.k, s["a"].stride(0), P(s["packed"].buf.data_ptr()), w.n,
                P(s["c"].data_ptr()), s["c"].stride(0), P(ws.data_ptr() if ws is not None else 0),
                ws.numel() if ws is not None else 0, P(stream.cuda_stream))
        for _ in range(5):
            lib.mxfp4_gemm(*argv)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            lib.mxfp4_gemm(*argv)
        dt = time.perf_counter() - t0
        torch.cuda.synchronize()
        out[w.name] = round(dt / calls * 1e6, 2)
    t0 = time.perf_counter()
    for _ in range(calls):
        lib.mxfp4_version()
    out["ctypes_call_floor"] = round((time.perf_counter() - t0) / calls * 1e6, 2)
    return out


# ------------------------------------------------------------ CPU oracle
def _bits(t):
    import numpy as np
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_of(w):
    """The bounded oracle sample of one shape: rows [0, ms) x weight rows
    (output columns) [0, ns): every row and the first 1/8 of the columns,
    the m=4096 shape only its first 1/16 of the rows."""
    ms = w.m if w.m < 4096 else w.m // 16
    return ms, max(1, w.n // 8)


def cpu_baseline(shapes, budget_s=12.0):
    """The oracle (quant of A, then the fp64 GEMM; single-threaded C) on the
    bounded sample of every shape, repeated until about `budget_s` seconds
    have been timed.  The first repetition doubles as the in-process parity
    check of the GPU run that preceded it: the oracle's quantization of B's
    sample rows against the bytes the library made, and the GPU's C against
    the oracle's on the sample at the stated tolerance."""
    import numpy as np

    import oracle
    prepared, parity = [], {}
    for s in shapes:
        w = s["w"]
        ms, ns = sample_of(w)
        bq, bs = oracle.quant(_bits(s["b_cpu"][:ns]))
        a_bits = _bits(s["a_cpu"][:ms])
        prepared.append((w, a_bits, bq, bs, ms, ns))
        parity[w.name] = {"b_quant_bit_exact": bool(np.array_equal(bq, s["bq_s"]) and np.array_equal(bs, s["bs_s"])),
                          "sample": f"rows [0,{ms}) x cols [0,{ns})"}
    total_t, total_b, reps = 0.0, 0, 0
    per_shape_t = {}
    while total_t < budget_s and reps < 1000:
        for (w, a_bits, bq, bs, ms, ns), s in zip(prepared, shapes):
            t0 = time.perf_counter()
            aq, a_s = oracle.quant(a_bits)
            ref = oracle.gemm(aq, a_s, bq, bs)
            dt = time.perf_counter() - t0
            total_t += dt
            total_b += algorithmic_bytes(ms, ns, w.k)
            per_shape_t.setdefault(w.name, []).append(dt)
            if reps == 0:
                got = s["c_first"][:ms, :ns]
                scale = float(np.max(np.abs(ref)))
                bound = REL_TOL * np.abs(ref) + ABS_TOL_FRAC * scale
                err = np.abs(got - ref)
                p = parity[w.name]
                p["max_err_over_bound"] = round(float(np.max(err / bound)), 4)
                p["finite"] = bool(np.all(np.isfinite(got)))
                p["ok"] = bool(p["finite"] and np.all(err <= bound) and p["b_quant_bit_exact"])
        reps += 1
    cores, model = host_cpu()
    base = {"value": round(total_b / total_t / 1e12, 9), "unit": "TB/s", "cores": 1, "kind": "oracle",
            "host_cores": cores, "cpu_model": model,
            "sample": f"{reps} x (oracle quant of A + fp64 GEMM on each shape's sample: every row x the first 1/8 "
                      f"of the output columns, m=4096 its first 1/16 of the rows), single-threaded C, "
                      f"{total_t:.1f} s",
            "per_shape_ms": {k: round(statistics.mean(v) * 1e3, 2) for k, v in per_shape_t.items()}}
    return base, parity


def _oracle_prepare(names, fraction):
    """Inputs for the reference arm's step: each shape's sample rows of A and
    the first `fraction` of its sample's weight rows, B quantized by the oracle."""
    import oracle
    from precision_bf16_mxfp4_gb300 import inputs
    prepared = []
    for nm in names:
        w = inputs.WORKLOADS[nm]
        a, b = inputs.make_inputs(nm, seed=0)
        ms, ns_full = sample_of(w)
        ns = max(1, int(round(ns_full * 8 * fraction)))
        bq, bs = oracle.quant(_bits(b[:ns]))
        prepared.append((w, _bits(a[:ms]), bq, bs, ms, ns))
    return prepared


def _oracle_run(prepared):
    """The oracle (quant of A, then the fp64 GEMM) on prepared inputs.
    Returns (seconds, algorithmic bytes covered)."""
    import oracle
    t0 = time.perf_counter()
    covered = 0
    for w, a_bits, bq, bs, ms, ns in prepared:
        aq, a_s = oracle.quant(a_bits)
        oracle.gemm(aq, a_s, bq, bs)
        covered += algorithmic_bytes(ms, ns, w.k)
    return time.perf_counter() - t0, covered


def oracle_step_sample(names, fraction):
    """The oracle on the first `fraction` of each shape's output columns."""
    return _oracle_run(_oracle_prepare(names, fraction))


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
    cores, model = host_cpu()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 9), "unit": "TB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": "+".join(names), "sample_fraction_of_columns": frac},
        "cpu_baseline": {"value": round(value, 9), "unit": "TB/s", "cores": 1, "kind": "oracle",
                         "host_cores": cores, "cpu_model": model,
                         "sample": f"oracle quant of A + fp64 GEMM per shape on its sample rows (every row; m=4096 "
                                   f"the first 1/16) x {frac:.5f} of the output columns, per step"},
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
    """The dense FP4 tensor-core rate: the median of `runs` launches of the
    library's microbenchmark, with the SM clocks sampled meanwhile."""
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
    """The launch floors of the small-m GEMMs: CUDA events around one empty
    kernel and around two back to back, and the same for minimal kernels
    (a global read, a tensor-memory allocation and a global write per CTA),
    each after the same L2 flush the GEMMs get (mean and median over
    `steps`, in microseconds)."""
    import torch

    import precision_bf16_mxfp4_gb300 as mx
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    flush = make_flush(dev)
    stream = torch.cuda.current_stream(dev)
    out = {"ctas": ctas, "steps": steps, "l2": "flushed before every timed launch (write of %d MiB)" %
           (flush.numel() >> 20)}
    for count in (1, 2):
        mean, med = event_time(stream, flush, lambda: mx.launch_empty(count, ctas, dev), steps, warmup)
        out[f"{count}_kernel_us"] = {"mean": round(mean * 1e6, 3), "median": round(med * 1e6, 3)}
        mean, med = event_time(stream, flush, lambda: mx.launch_minimal(count, ctas, dev), steps, warmup)
        out[f"{count}_minimal_kernel_us"] = {"mean": round(mean * 1e6, 3), "median": round(med * 1e6, 3)}
    return out


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
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
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
