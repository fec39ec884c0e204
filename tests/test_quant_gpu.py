"""GPU parity of mxfp4_quant against the oracle: bit-exact nibbles and scale bytes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import precision_bf16_mxfp4_gb300 as mx
from precision_bf16_mxfp4_gb300 import inputs
from tests.helpers import bf16_bits, from_bits

pytestmark = pytest.mark.gpu


def _gpu_quant(a_cpu: torch.Tensor, lda: int | None = None):
    m, k = a_cpu.shape
    if lda is not None and lda != k:
        big = torch.full((m, lda), float("nan"), dtype=torch.bfloat16)
        big[:, :k] = a_cpu
        a_dev = big.cuda()[:, :k]
    else:
        a_dev = a_cpu.cuda()
    q, s = mx.quant(a_dev)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _check(a_cpu: torch.Tensor, lda: int | None = None):
    q, s = _gpu_quant(a_cpu, lda)
    rq, rs = oracle.quant(bf16_bits(a_cpu))
    bad_s = np.argwhere(s != rs)
    assert bad_s.size == 0, f"scale mismatch at {bad_s[:5].tolist()}: gpu {s[tuple(bad_s[0])]} oracle {rs[tuple(bad_s[0])]}"
    bad_q = np.argwhere(q != rq)
    assert bad_q.size == 0, f"nibble mismatch at {bad_q[:5].tolist()}: gpu {q[tuple(bad_q[0])]:#04x} oracle {rq[tuple(bad_q[0])]:#04x}"


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_quant_workload_activations(name):
    w = inputs.WORKLOADS[name]
    if w.m * w.k > 4096 * 2048:
        pytest.skip("too large")
    a, _ = inputs.make_inputs(name)
    _check(a)


@pytest.mark.parametrize("name", ["m4_n2880_k512", "m16_n2112_k7168"])
def test_quant_workload_weights(name):
    _, b = inputs.make_inputs(name)
    _check(b)


def test_quant_every_finite_bf16_value():
    bits = inputs.all_finite_bf16_bits().numpy().view(np.uint16)
    rng = np.random.default_rng(0)
    perm = rng.permutation(bits.size)
    pad = (-bits.size) % 512
    arr = np.concatenate([bits[perm], np.zeros(pad, np.uint16)]).reshape(-1, 512)
    _check(from_bits(arr))


def test_quant_every_block_exponent():
    """For each anchor magnitude (every finite bf16 exponent and several
    mantissas), a block of the anchor plus 31 random smaller values."""
    rng = np.random.default_rng(1)
    rows = []
    for exp_field in range(0, 255):
        for mant in (0x00, 0x3F, 0x40, 0x5F, 0x60, 0x7F):
            anchor = (exp_field << 7) | mant
            if anchor == 0:
                continue
            blk = np.zeros(32, np.uint16)
            lo_e = rng.integers(max(0, exp_field - 12), exp_field + 1, 31)
            m_ = rng.integers(0, 128, 31)
            other = (lo_e << 7) | m_
            other = np.minimum(other, anchor)
            sign = rng.integers(0, 2, 31) << 15
            blk[1:] = other | sign
            blk[0] = anchor | (rng.integers(0, 2) << 15)
            rng.shuffle(blk)
            rows.append(blk)
    while len(rows) % 8:
        rows.append(np.zeros(32, np.uint16))
    arr = np.stack(rows).reshape(-1, 256)
    _check(from_bits(arr))


def test_quant_every_value_under_every_block_exponent():
    """Exhaustive encoder check: for every finite bf16 anchor exponent and two
    anchor mantissas (0x5F stays in its binade after the +0x200000 rounding,
    0x7F rounds up into the next), every bf16 value of magnitude up to the
    anchor's, both signs, in blocks led by the anchor (about 16.6 M values).
    Every (element, block exponent) pair the quantizer can meet is covered,
    including products far below the fp32 normal range."""
    groups = []
    for exp_field in range(0, 255):
        for mant in (0x5F, 0x7F):
            anchor = (exp_field << 7) | mant
            mags = np.arange(0, anchor + 1, dtype=np.uint32)
            vals = np.concatenate([mags, mags | 0x8000]).astype(np.uint16)
            pad = (-vals.size) % 31
            vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 31)
            lead = np.full((vals.shape[0], 1), anchor, np.uint16)
            groups.append(np.concatenate([lead, vals], axis=1))
    blocks = np.concatenate(groups)
    pad = (-blocks.shape[0]) % 32
    blocks = np.concatenate([blocks, np.zeros((pad, 32), np.uint16)])
    arr = blocks.reshape(-1, 1024)
    _check(from_bits(arr))


def test_quant_special_blocks():
    blocks = [
        np.zeros(32, np.uint16),                                   # all +0 -> e8m0 0
        np.full(32, 0x8000, np.uint16),                            # all -0 -> nibbles 0x8
        np.full(32, 0x7F7F, np.uint16),                            # bf16 max -> exponent field 255
        np.full(32, 0x0001, np.uint16),                            # smallest subnormal
        np.arange(32, dtype=np.uint16) | 0x0040,                   # subnormal range
        np.array([0x3F80] + [0xBD4D] * 31, np.uint16),             # -0.05 next to 1.0: negative zeros
        np.array([0x4220, 0x3F80] + [0] * 30, np.uint16),          # outlier tie 5.0
    ]
    arr = np.stack(blocks + [np.zeros(32, np.uint16)]).reshape(1, -1)
    _check(from_bits(arr))


@pytest.mark.parametrize("m,k,lda", [(1, 32, 32), (3, 96, 96), (5, 288, 296), (7, 544, 552), (130, 480, 512),
                                     (1, 7168, 7168), (257, 256, 264)])
def test_quant_ragged_shapes(m, k, lda):
    a = inputs.random_bf16(m, k, seed=m * 1000 + k, std=3.0)
    _check(a, lda=lda)


@pytest.mark.parametrize("m,k,lda", [(32768, 4096, 4096), (3, 262144, 262144), (65536, 64, 72)])
def test_quant_largest_shapes(m, k, lda):
    # far beyond the workloads: 134 M elements; rows of 8192 blocks; 65536
    # rows of two blocks with a padded stride - every byte against the oracle
    a = inputs.random_bf16(m, k, seed=m + k, std=3.0)
    _check(a, lda=lda)


def test_quant_empty_is_a_noop():
    a = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    q, s = mx.quant(a)
    assert q.shape == (0, 32) and s.shape == (0, 2)


def test_quant_matches_on_a_side_stream():
    a = inputs.random_bf16(64, 1024, seed=5)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        q, s = mx.quant(a.cuda())
    stream.synchronize()
    rq, rs = oracle.quant(bf16_bits(a))
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
