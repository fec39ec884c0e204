"""Shared test helpers (seeded inputs, tolerance, marshalling)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# |gpu - ref| <= 2^-7 |ref| + 1e-3 max|ref|: products of e2m1 values and
# power-of-two scales are exact, so only the fp32 summation order inside the
# tensor cores and the final bf16 rounding (relative 2^-9) differ from the
# exact fp64 reference.
REL_TOL = 2.0 ** -7
ABS_TOL_FRAC = 1e-3


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def assert_close_to_ref(got: np.ndarray, ref: np.ndarray, scale: float | None = None, what: str = ""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    s = float(np.max(np.abs(ref))) if scale is None else scale
    bound = REL_TOL * np.abs(ref) + ABS_TOL_FRAC * s
    err = np.abs(got - ref)
    bad = np.nonzero(err > bound)
    if bad[0].size:
        idx = tuple(b[0] for b in bad)
        raise AssertionError(f"{what}: {bad[0].size} entries out of tolerance; first at {idx}: "
                             f"got {got[idx]!r} ref {ref[idx]!r} bound {bound[idx]!r}")


def oracle_weights(b_bf16: torch.Tensor):
    """B quantized by the oracle (as the workloads specify), as numpy arrays."""
    return oracle.quant(bf16_bits(b_bf16))


def packed_from_oracle(b_bf16: torch.Tensor, device="cuda"):
    import precision_bf16_mxfp4_gb300 as mx
    bq, bs = oracle_weights(b_bf16)
    packed = mx.prepack_b(torch.from_numpy(bq).to(device), torch.from_numpy(bs).to(device))
    return packed, bq, bs


def gloo_max_over_ranks_worker(rank: int, world: int, port: int, values, out_queue):
    """Child of the 2-rank gloo test: bench.py's barrier and max-over-ranks."""
    import os
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.max_over_ranks(values[rank], world)
        bench.barrier(world)
        out_queue.put((rank, got))
    finally:
        dist.destroy_process_group()
