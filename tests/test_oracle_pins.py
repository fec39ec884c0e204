"""Pins for the CPU oracle, each against something other than the oracle itself.

* hand-worked examples (tests/golden/quant_examples.txt), worked from the block
  rule of the "kernelbot amd-mxfp4-mm" pages (submission 694791, "MXFP4
  quantization"; submission 752099, `_bf16_to_fp4_hw`);
* the e2m1 value set from the format's own definition (sign, 2-bit exponent
  with bias 1, 1-bit mantissa, subnormal when the exponent field is 0);
* a closed form of the block exponent (frexp plus the 1.75 round-up boundary),
  over every finite bf16 magnitude;
* an independent threshold formulation of round-to-nearest-even onto the e2m1
  grid, over every finite bf16 value times every block exponent;
* losslessness, sign symmetry and monotonicity properties;
* exact rational brute force of the GEMM and its reduction to a plain matmul.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_examples.txt")


def _bf16_value(bits: int) -> float:
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


def _format_value(nibble: int) -> float:
    """e2m1 by its definition: s | e1 e0 | m, bias 1, subnormal at e = 0."""
    s = (nibble >> 3) & 1
    e = (nibble >> 1) & 3
    mant = nibble & 1
    mag = mant * 0.5 if e == 0 else (1.0 + 0.5 * mant) * 2.0 ** (e - 1)
    return -mag if s else mag


def _parse_golden():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fields = dict(f.split("=", 1) for f in line.split())

        def pairs(txt, conv):
            out = {}
            for item in filter(None, txt.split(",")):
                i, v = item.split(":")
                out[int(i)] = conv(v)
            return out

        cases.append(dict(
            values=pairs(fields["values"], lambda v: int(v, 16)),
            ub=int(fields["ub"]), e8m0=int(fields["e8m0"]),
            nibbles=pairs(fields["nibbles"], lambda v: int(v, 16)),
            deq=pairs(fields["deq"], float)))
    return cases


GOLDEN_CASES = _parse_golden()


def test_golden_file_is_nonempty():
    assert len(GOLDEN_CASES) >= 14


@pytest.mark.parametrize("case", GOLDEN_CASES, ids=lambda c: str(sorted(c["values"].items()))[:40])
def test_golden_quant_examples(case):
    block = np.zeros((1, 32), np.uint16)
    for i, b in case["values"].items():
        block[0, i] = b
    assert oracle.block_exponent(block[0]) == case["ub"]
    q, s = oracle.quant(block)
    assert s[0, 0] == case["e8m0"]
    nib = np.zeros(32, np.int64)
    nib[0::2] = q[0] & 0xF
    nib[1::2] = q[0] >> 4
    want = np.zeros(32, np.int64)
    for i, v in case["nibbles"].items():
        want[i] = v
    np.testing.assert_array_equal(nib, want)
    deq = oracle.dequant(q, s)[0]
    want_deq = np.zeros(32)
    for i, v in case["deq"].items():
        want_deq[i] = v
    np.testing.assert_array_equal(deq, want_deq)
    for i, v in case["deq"].items():  # signed zeros too
        assert math.copysign(1.0, deq[i]) == math.copysign(1.0, v)


def test_value_set_matches_format_definition():
    codes = np.arange(16, dtype=np.uint8)
    q = (codes[0::2] | (codes[1::2] << 4)).reshape(1, 8)
    q = np.concatenate([q, np.zeros((1, 8), np.uint8)], axis=1)  # pad to k = 32
    s = np.full((1, 1), 127, np.uint8)
    deq = oracle.dequant(q, s)[0, :16]
    want = [_format_value(c) for c in range(16)]
    np.testing.assert_array_equal(deq, want)
    assert sorted(set(abs(v) for v in deq)) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert math.copysign(1.0, deq[8]) == -1.0  # code 0x8 is negative zero


def _closed_form_ub(amax: float) -> int:
    """floor(log2 amax) - 2, plus one when amax >= 1.75 * 2^floor(log2 amax)."""
    if amax == 0.0:
        return -127
    mant, exp = math.frexp(amax)      # amax = mant * 2^exp, mant in [0.5, 1)
    e = exp - 1                       # floor(log2 amax), exact
    ub = e - 2 + (1 if amax >= 1.75 * 2.0 ** e else 0)
    return max(-127, min(127, ub))


def test_block_exponent_closed_form_every_bf16():
    for bits in range(0, 0x7F80):     # every finite non-negative bf16
        amax = _bf16_value(bits)
        want = _closed_form_ub(amax)
        assert oracle.block_exponent(np.array([bits], np.uint16)) == want, hex(bits)
        assert oracle.block_exponent(np.array([bits | 0x8000], np.uint16)) == want, hex(bits)


def test_block_exponent_uses_the_block_maximum():
    rng = np.random.default_rng(1)
    for _ in range(300):
        vals = (rng.standard_normal(32) * 2.0 ** rng.integers(-20, 20)).astype(np.float32)
        bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
        amax = max(abs(_bf16_value(int(b))) for b in bits)
        assert oracle.block_exponent(bits) == _closed_form_ub(amax)


def _threshold_code(q: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even onto {0,.5,1,1.5,2,3,4,6} written as comparisons
    with the midpoints; a midpoint goes to the neighbour with the even code."""
    return ((q > 0.25).astype(np.int64) + (q >= 0.75) + (q > 1.25) + (q >= 1.75)
            + (q > 2.5) + (q >= 3.5) + (q > 5.0))


def test_encode_exhaustive_against_thresholds():
    bits = np.arange(0, 65536, dtype=np.uint32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    bits = bits[finite].astype(np.uint16)
    mag = np.abs((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    sign = (bits >> 15).astype(np.int64)
    for ub in range(-127, 128):
        q = np.ldexp(mag, -ub)
        want = _threshold_code(q) | (sign << 3)
        got = oracle.encode_many(bits, np.full(bits.shape, ub, np.int32))
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (ub, hex(int(bits[bad[0]])), int(got[bad[0]]), int(want[bad[0]]))


def test_quant_layout_two_blocks():
    # block 0 all 1.0 -> ub -2 (e8m0 125), q = 4 -> code 6 in both nibbles;
    # block 1 all 3.0 -> amax 1.5 * 2 (fraction .5, no round-up) -> ub -1 (e8m0 126), q = 6 -> code 7
    row = np.concatenate([np.full(32, 0x3F80, np.uint16), np.full(32, 0x4040, np.uint16)])
    row[33] = 0xC040  # -3.0 at an odd index of block 1 -> high nibble of byte 16 is 0xF
    q, s = oracle.quant(row.reshape(1, 64))
    assert list(s[0]) == [125, 126]
    assert all(b == 0x66 for b in q[0, :16])
    assert q[0, 16] == 0xF7
    assert all(b == 0x77 for b in q[0, 17:])


def test_quant_rows_are_independent():
    a = torch.randn(5, 96, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    q, s = oracle.quant(a)
    for i in range(5):
        qi, si = oracle.quant(a[i:i + 1])
        np.testing.assert_array_equal(q[i], qi[0])
        np.testing.assert_array_equal(s[i], si[0])


def test_lossless_on_scaled_grid_values():
    rng = np.random.default_rng(7)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    nblocks = 100_000
    s_exp = rng.integers(-127, 126, nblocks)
    g = grid[rng.integers(0, 8, (nblocks, 32))]
    sign = np.where(rng.random((nblocks, 32)) < 0.5, -1.0, 1.0)
    vals = (g * sign) * np.ldexp(1.0, s_exp)[:, None]
    f32 = vals.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), vals)  # representable
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(((bits.astype(np.uint32) << 16).view(np.float32)).astype(np.float64), vals)
    q, s = oracle.quant(bits.reshape(nblocks, 32))
    deq = oracle.dequant(q, s)
    np.testing.assert_array_equal(np.abs(deq), np.abs(vals))


def test_lossy_below_the_clamp():
    # 0.5 * 2^-128 = 2^-129: ub would be -130 but clamps to -127, q = 0.25 ties to 0
    bits = np.zeros((1, 32), np.uint16)
    bits[0, 0] = 0x0010  # 16 * 2^-133 = 2^-129 (bf16 subnormal)
    assert _bf16_value(0x0010) == 2.0 ** -129
    q, s = oracle.quant(bits)
    assert s[0, 0] == 0 and q[0, 0] == 0


def test_sign_symmetry_and_monotonicity():
    a = torch.randn(64, 256, generator=torch.Generator().manual_seed(11)).to(torch.bfloat16)
    q, s = oracle.quant(a)
    qn, sn = oracle.quant(-a)
    np.testing.assert_array_equal(s, sn)
    np.testing.assert_array_equal(q ^ 0x88, qn)
    deq = np.abs(oracle.dequant(q, s))
    x = np.abs(a.float().numpy().astype(np.float64))
    for i in range(64):
        for b in range(256 // 32):
            xs, ds = x[i, b * 32:(b + 1) * 32], deq[i, b * 32:(b + 1) * 32]
            order = np.argsort(xs, kind="stable")
            assert np.all(np.diff(ds[order]) >= 0)


def _random_mxfp4(rng, rows, k, lo=120, hi=134):
    q = rng.integers(0, 256, (rows, k // 2), dtype=np.uint8)
    s = rng.integers(lo, hi + 1, (rows, k // 32), dtype=np.uint8)
    return q, s


def _exact_value(q, s, i, j):
    byte = int(q[i, j // 2])
    nib = byte & 0xF if j % 2 == 0 else byte >> 4
    return Fraction(_format_value(nib)) * Fraction(2) ** (int(s[i, j // 32]) - 127)


def test_gemm_exact_rational_bruteforce():
    rng = np.random.default_rng(5)
    m, n, k = 3, 5, 96
    aq, a_s = _random_mxfp4(rng, m, k)
    bq, b_s = _random_mxfp4(rng, n, k)
    c = oracle.gemm(aq, a_s, bq, b_s)
    assert c.shape == (m, n)
    for i in range(m):
        for j in range(n):
            exact = sum(_exact_value(aq, a_s, i, t) * _exact_value(bq, b_s, j, t) for t in range(k))
            assert Fraction(c[i, j]) == exact, (i, j)


def test_gemm_reduces_to_plain_matmul_at_unit_scale():
    rng = np.random.default_rng(9)
    m, n, k = 7, 6, 128
    aq, _ = _random_mxfp4(rng, m, k)
    bq, _ = _random_mxfp4(rng, n, k)
    ones_a = np.full((m, k // 32), 127, np.uint8)
    ones_b = np.full((n, k // 32), 127, np.uint8)
    dec = np.vectorize(_format_value)
    a_val = np.zeros((m, k))
    a_val[:, 0::2] = dec(aq & 0xF)
    a_val[:, 1::2] = dec(aq >> 4)
    b_val = np.zeros((n, k))
    b_val[:, 0::2] = dec(bq & 0xF)
    b_val[:, 1::2] = dec(bq >> 4)
    want = torch.matmul(torch.from_numpy(a_val), torch.from_numpy(b_val).T).numpy()
    np.testing.assert_array_equal(oracle.gemm(aq, ones_a, bq, ones_b), want)


def test_gemm_entries_and_dequant_path_agree_with_gemm():
    rng = np.random.default_rng(13)
    m, n, k = 9, 11, 160
    aq, a_s = _random_mxfp4(rng, m, k)
    bq, b_s = _random_mxfp4(rng, n, k)
    c = oracle.gemm(aq, a_s, bq, b_s)
    rows = rng.integers(0, m, 40)
    cols = rng.integers(0, n, 40)
    np.testing.assert_array_equal(oracle.gemm_entries(aq, a_s, bq, b_s, rows, cols), c[rows, cols])
    np.testing.assert_allclose(oracle.gemm_via_dequant(aq, a_s, bq, b_s), c, rtol=1e-12, atol=0)
