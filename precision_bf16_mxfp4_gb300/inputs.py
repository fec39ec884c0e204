"""Seeded synthetic inputs for the MXFP4 GEMM workloads.

This module only draws random numbers; it holds none of the method's
arithmetic (no quantization, no scaling rule, no packing), so that the CUDA
path and the CPU oracle can both be fed from it without sharing any of the
computation they are compared on.

The shapes are the ones the "kernelbot amd-mxfp4-mm" submission pages
benchmark (submission 752099, module docstring listing the benchmark shapes, plus the compute-bound large-M case); the value distributions follow
the workload recipe stated for each shape below.  The leaderboard's own data
generator is not available, so these seeded draws stand in for it.

Every workload draws A first, then B, then any auxiliary tensors, from one
``torch.Generator`` seeded with ``seed`` (default 0).  Normal draws are fp32
converted to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    m: int
    n: int
    k: int
    a_kind: str      # "normal", "block_exp_zero", "outliers"
    b_std: float
    note: str


WORKLOADS = {
    "m4_n2880_k512": Workload("m4_n2880_k512", 4, 2880, 512, "normal", 1.0,
                              "small m, single-pass K"),
    "m32_n4096_k512": Workload("m32_n4096_k512", 32, 4096, 512, "normal", 1.0,
                               "single-pass K, fused in-register quant"),
    "m32_n2880_k512": Workload("m32_n2880_k512", 32, 2880, 512, "normal", 1.0,
                               "single-pass K, fused in-register quant"),
    "m16_n2112_k7168": Workload("m16_n2112_k7168", 16, 2112, 7168, "block_exp_zero", 0.02,
                                "thin grid, long K: split-K"),
    "m64_n7168_k2048": Workload("m64_n7168_k2048", 64, 7168, 2048, "outliers", 0.02,
                                "0.1% outliers exercise saturation"),
    "m256_n3072_k1536": Workload("m256_n3072_k1536", 256, 3072, 1536, "normal", 0.02,
                                 "separate quant kernel + GEMM on quantized A"),
    "m4096_n7168_k2048": Workload("m4096_n7168_k2048", 4096, 7168, 2048, "normal", 0.02,
                                  "compute-heavy, separate quant + GEMM"),
}

# The test shapes listed beside the benchmark shapes in the kernelbot
# amd-mxfp4-mm submission 752099 page (its per-shape configuration table):
# parity cases only, with the benchmark shapes' plain N(0,1) / N(0,0.02) inputs.
TEST_SHAPES = {
    "m8_n2112_k7168": Workload("m8_n2112_k7168", 8, 2112, 7168, "normal", 0.02, "thin, long K: split-K"),
    "m16_n3072_k1536": Workload("m16_n3072_k1536", 16, 3072, 1536, "normal", 0.02, "fused, medium K"),
    "m64_n3072_k1536": Workload("m64_n3072_k1536", 64, 3072, 1536, "normal", 0.02, "quant image + swap-AB"),
    "m256_n2880_k512": Workload("m256_n2880_k512", 256, 2880, 512, "normal", 0.02, "quant image + plain GEMM"),
}

# The pair of shapes the headline metric is quoted on (m=32, k=512).
HEADLINE = ("m32_n4096_k512", "m32_n2880_k512")


def _normal(gen: torch.Generator, rows: int, cols: int, std: float) -> torch.Tensor:
    return (torch.randn(rows, cols, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


def make_a(w: Workload, gen: torch.Generator) -> torch.Tensor:
    """Activation matrix A, bf16 [m, k], drawn per the workload's recipe."""
    x = torch.randn(w.m, w.k, generator=gen, dtype=torch.float32)
    if w.a_kind == "normal":
        pass
    elif w.a_kind == "block_exp_zero":
        # each 32-element K block multiplied by 2^u, u uniform in {-8..8};
        # each block zeroed with probability 1/64
        nb = w.k // 32
        u = torch.randint(-8, 9, (w.m, nb), generator=gen).to(torch.float32)
        zero = torch.rand(w.m, nb, generator=gen) < (1.0 / 64.0)
        mult = torch.pow(2.0, u) * (~zero).to(torch.float32)
        x = (x.view(w.m, nb, 32) * mult[:, :, None]).view(w.m, w.k)
    elif w.a_kind == "outliers":
        # 0.1% of entries replaced by +-U(8, 64), sign with probability 1/2
        pick = torch.rand(w.m, w.k, generator=gen) < 1e-3
        mag = 8.0 + 56.0 * torch.rand(w.m, w.k, generator=gen)
        sign = torch.where(torch.rand(w.m, w.k, generator=gen) < 0.5, -1.0, 1.0)
        x = torch.where(pick, mag * sign, x)
    else:
        raise ValueError(w.a_kind)
    return x.to(torch.bfloat16)


def make_inputs(name_or_workload, seed: int = 0):
    """Return (A bf16 [m,k], B bf16 [n,k]) on the CPU for one workload."""
    if isinstance(name_or_workload, str):
        w = WORKLOADS[name_or_workload] if name_or_workload in WORKLOADS else TEST_SHAPES[name_or_workload]
    else:
        w = name_or_workload
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    a = make_a(w, gen)
    b = _normal(gen, w.n, w.k, w.b_std)
    return a, b


def random_bf16(rows: int, cols: int, seed: int, std: float = 1.0) -> torch.Tensor:
    """A plain N(0, std^2) bf16 matrix for tests of arbitrary shape."""
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    return _normal(gen, rows, cols, std)


def all_finite_bf16_bits() -> torch.Tensor:
    """Every finite bf16 bit pattern (65,280 of them), as int16 bits."""
    bits = torch.arange(0, 65536, dtype=torch.int32)
    exp = (bits >> 7) & 0xFF
    return bits[exp != 0xFF].to(torch.int16)
