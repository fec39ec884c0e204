/*
 * MXFP4 oracle: a plain, slow, single-threaded CPU restatement of what the
 * MXFP4 GEMM  C[m,n] = quant(A) . B^T  computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file; only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark use it.
 * It shares no code, header, table or constant with the CUDA sources.
 *
 * Sources, all on the "kernelbot amd-mxfp4-mm" submission pages:
 *   - block scale rule: submission 694791, "MXFP4 quantization:
 *     bf16 -> fp4(e2m1) + e8m0 block scales", the amax / round-up / -2 /
 *     clamp / +127 steps; submission 752099 `_bf16_to_fp4_hw`,
 *     which reads the exponent field instead of taking floor(log2);
 *   - element encoding: submission 694791, same section: scale the element by
 *     2^(-ub), round to the e2m1 grid with ties to even, saturate at 6.0,
 *     keep the sign as bit 3;
 *   - packing: submission 694791, same section: two codes per byte, even K index in
 *     the low nibble;
 *   - GEMM semantics: submission 752099 `tl.dot_scaled(a, a_scale, "e2m1", b,
 *     b_scale, "e2m1", acc)` -- a dequantize-then-multiply product.
 *
 * Arithmetic is fp64 throughout.  Every quantity the quantizer forms is
 * exact in fp64 (bf16 inputs have 8 significant bits, scales are powers of
 * two), so the code chosen for an element is the mathematically nearest
 * grid point; the e2m1 rounding is written as a nearest-grid search, not as
 * the bit manipulation the pages use.  The GEMM sums exact products in
 * fp64 with no blocking or reordering.
 *
 * Readings where the pages leave a step open:
 *   - the scale exponent is read from the fp32 exponent field of the
 *     rounded amax (three of the four page variants), not floor(log2());
 *     they differ only when the rounded amax overflows to infinity;
 *   - an e8m0 byte of 0 means 2^-127, not zero;
 *   - a negative element that rounds to zero keeps its sign: nibble 0x8;
 *   - subnormal bf16 inputs are taken at their exact value (no flush);
 *   - NaN and infinite inputs are outside the method and not defined here.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* The eight non-negative e2m1 magnitudes, indexed by the 3-bit code
 * (exponent bits 2..1, mantissa bit 0).  Submission 694791, "MXFP4 quantization". */
static const double kGrid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Unbiased block exponent ub for one 32-element block of bf16 values.
 * amax is widened to fp32 (exact); its bit pattern gets +0x200000 and is
 * masked with 0xFF800000, which rounds the magnitude up to the next power
 * of two when its fraction is >= 0.75; ub = exponent field - 127 - 2,
 * clamped to [-127, 127].  Submission 694791 "MXFP4 quantization" (amax, round-up,
 * the -2 that puts the block maximum at or below the top of the e2m1 range, clamp); submission 752099
 * `_bf16_to_fp4_hw` for the exponent-field form. */
int oracle_block_exponent(const uint16_t *x, int64_t count)
{
    double amax = 0.0;
    for (int64_t i = 0; i < count; ++i) {
        double v = fabs(bf16_value(x[i]));
        if (v > amax)
            amax = v;
    }
    float amax_f = (float)amax; /* exact: amax is a bf16 value */
    uint32_t bits;
    memcpy(&bits, &amax_f, sizeof bits);
    uint32_t rounded = (bits + 0x200000u) & 0xFF800000u;
    int ub = (int)((rounded >> 23) & 0xFFu) - 127 - 2;
    if (ub < -127)
        ub = -127;
    if (ub > 127)
        ub = 127;
    return ub;
}

/* e2m1 magnitude code (0..7) of a non-negative real q.  Values at or above
 * the largest finite e2m1 value saturate to it (code 7, 6.0); below that,
 * the code is the index of the nearest grid value, ties to the even code.
 * Submission 694791 "MXFP4 quantization" (saturate at >= 6, round to nearest even).
 * For q < 6 every distance below is exact in fp64 whenever it matters: q has
 * at most 8 significant bits, so q - g is exact for q >= 2^-40, and smaller q
 * are unambiguously nearest to 0. */
int oracle_e2m1_code(double q)
{
    if (q >= 6.0)
        return 7;
    int best = 0;
    double best_d = fabs(q - kGrid[0]);
    for (int c = 1; c < 8; ++c) {
        double d = fabs(q - kGrid[c]);
        if (d < best_d || (d == best_d && (c % 2) == 0 && (best % 2) != 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* 4-bit e2m1 nibble of one element given the block exponent ub:
 * q = x * 2^-ub (exact in fp64), magnitude code from the nearest-grid
 * search, sign of x in bit 3 (kept for values that round to zero). */
int oracle_encode(uint16_t x, int ub)
{
    double v = bf16_value(x);
    double q = ldexp(fabs(v), -ub);
    int code = oracle_e2m1_code(q);
    int sign = (x >> 15) & 1;
    return code | (sign << 3);
}

/* Quantize A (bf16 [m,k], row stride lda elements) to MXFP4:
 *   q     [m, k/2]  u8, byte j of a row = code(2j) | code(2j+1) << 4
 *   scale [m, k/32] u8, e8m0 = ub + 127
 * k must be a multiple of 32.  Submission 694791 "MXFP4 quantization" (per-32 block
 * scale, packing `ev | od << 4`). */
void oracle_quant(const uint16_t *a, int64_t m, int64_t k, int64_t lda,
                  uint8_t *q, uint8_t *scale)
{
    int64_t nblk = k / 32;
    for (int64_t i = 0; i < m; ++i) {
        const uint16_t *row = a + i * lda;
        for (int64_t b = 0; b < nblk; ++b) {
            const uint16_t *blk = row + b * 32;
            int ub = oracle_block_exponent(blk, 32);
            scale[i * nblk + b] = (uint8_t)(ub + 127);
            for (int t = 0; t < 32; t += 2) {
                int lo = oracle_encode(blk[t], ub);
                int hi = oracle_encode(blk[t + 1], ub);
                q[i * (k / 2) + b * 16 + t / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* Value of one element of an MXFP4 matrix: (-1)^s * grid[code] *
 * 2^(e8m0 - 127).  An e8m0 byte of 0 is 2^-127. */
static double element_value(const uint8_t *q, const uint8_t *scale,
                            int64_t k, int64_t row, int64_t col)
{
    uint8_t byte = q[row * (k / 2) + col / 2];
    int nib = (col % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    double mag = kGrid[nib & 7];
    double s = ldexp(1.0, (int)scale[row * (k / 32) + col / 32] - 127);
    double v = mag * s;
    return (nib & 8) ? -v : v;
}

/* Dequantize MXFP4 [r, k] to fp64 [r, k]. */
void oracle_dequant(const uint8_t *q, const uint8_t *scale, int64_t r,
                    int64_t k, double *out)
{
    for (int64_t i = 0; i < r; ++i)
        for (int64_t j = 0; j < k; ++j)
            out[i * k + j] = element_value(q, scale, k, i, j);
}

/* One output of the GEMM: sum over k of deq(A)[i,kk] * deq(B)[j,kk],
 * in fp64, in order of kk. */
static double gemm_entry(const uint8_t *aq, const uint8_t *as,
                         const uint8_t *bq, const uint8_t *bs, int64_t k,
                         int64_t i, int64_t j)
{
    double acc = 0.0;
    for (int64_t kk = 0; kk < k; ++kk)
        acc += element_value(aq, as, k, i, kk) * element_value(bq, bs, k, j, kk);
    return acc;
}

/* C[m,n] = deq(A) . deq(B)^T in fp64.  A: q [m,k/2] + scale [m,k/32];
 * B: q [n,k/2] + scale [n,k/32].  Submission 752099 `tl.dot_scaled` semantics. */
void oracle_gemm(const uint8_t *aq, const uint8_t *as, const uint8_t *bq,
                 const uint8_t *bs, int64_t m, int64_t n, int64_t k,
                 double *c)
{
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < n; ++j)
            c[i * n + j] = gemm_entry(aq, as, bq, bs, k, i, j);
}

/* The same GEMM evaluated only at (rows[t], cols[t]), t < count. */
void oracle_gemm_entries(const uint8_t *aq, const uint8_t *as,
                         const uint8_t *bq, const uint8_t *bs, int64_t k,
                         const int64_t *rows, const int64_t *cols,
                         int64_t count, double *out)
{
    for (int64_t t = 0; t < count; ++t)
        out[t] = gemm_entry(aq, as, bq, bs, k, rows[t], cols[t]);
}

/* oracle_encode applied to count (x, ub) pairs; for exhaustive checks. */
void oracle_encode_many(const uint16_t *x, const int32_t *ub, int64_t count,
                        uint8_t *out)
{
    for (int64_t t = 0; t < count; ++t)
        out[t] = (uint8_t)oracle_encode(x[t], ub[t]);
}
