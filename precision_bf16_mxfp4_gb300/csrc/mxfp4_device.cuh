// Device-side building blocks shared by the MXFP4 kernels: the block-scale
// rule, the e2m1 encoder, and the tiled operand image that the tcgen05 MMA
// reads through bulk copies.
//
// Quantization rule (kernelbot amd-mxfp4-mm, submission 694791, "MXFP4
// quantization: bf16 -> fp4(e2m1) + e8m0 block scales"; exponent-field form
// as in submission 752099 `_bf16_to_fp4_hw`):
//   amax over 32 consecutive K elements; u = (fp32 bits of amax + 0x200000)
//   & 0xFF800000; ub = clamp(exponent field of u - 129, -127, 127);
//   e8m0 = ub + 127; each element x -> e2m1(x * 2^-ub) rounded to nearest
//   even on the grid {0,.5,1,1.5,2,3,4,6}, saturating at 6, sign in bit 3;
//   two codes per byte, even K index in the low nibble.
#pragma once
#include <cstdint>

namespace mxfp4 {

// ------------------------------------------------------------ image layout
// An MXFP4 matrix X[R, K] is stored for the MMA as blocks of 128 rows x 256 K
// elements.  Block (rt, kt) sits at (rt * KT + kt) * 17408 bytes, so the K
// blocks of one row tile are contiguous and a single bulk copy can move
// several of them.  Each block holds
//   bytes [0, 16384): 128 rows of 128 bytes in the 128-byte-swizzled K-major
//     order the MMA descriptor expects (16-byte chunk c of row r sits at
//     chunk c ^ (r & 7));
//   bytes [16384, 17408): the e8m0 scales as two 512-byte atoms (K blocks
//     0-3, 4-7); inside an atom, row r and block b sit at
//     (r % 32) * 16 + (r / 32) * 4 + b, the 32-lane x 16-byte shape of a
//     tensor-memory lane quadrant's scale columns (the kernels store each
//     atom row into its lane with tcgen05.st).
// Rows beyond R and K beyond the matrix are zero in the weight image.
constexpr int kTileRows = 128;
constexpr int kTileK = 256;
constexpr int kTileDataBytes = 16384;
constexpr int kTileSfBytes = 1024;
constexpr int kTileBytes = kTileDataBytes + kTileSfBytes;  // 17 x 1024: blocks stay 1024-byte aligned
constexpr int kAtomBytes = 512;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

__host__ __device__ inline int64_t image_bytes(int64_t rows, int64_t k) {
  return ceil_div(rows, kTileRows) * ceil_div(k, kTileK) * kTileBytes;
}
// offset of block (rt, kt) in an image with kt_count K blocks per row tile
__host__ __device__ inline int64_t image_block(int64_t rt, int64_t kt, int64_t kt_count) {
  return (rt * kt_count + kt) * kTileBytes;
}
// byte of row r (0..127), packed-K byte kb (0..127) inside a data tile
__host__ __device__ inline int tile_data_offset(int r, int kbyte) {
  return r * 128 + ((((kbyte >> 4) ^ (r & 7)) & 7) << 4) + (kbyte & 15);
}
// scale byte of row r (0..127), K block b (0..7) inside a scale tile
__host__ __device__ inline int tile_sf_offset(int r, int b) {
  return ((b >> 2) * kAtomBytes) + ((r & 31) << 4) + ((r >> 5) << 2) + (b & 3);
}

// ------------------------------------------------------------ quantization
// Largest |x| among the 32 bf16 values of one block, as a 15-bit magnitude
// pattern (for finite values the pattern order is the magnitude order).
__device__ __forceinline__ uint32_t absmax32_bits(const uint4 (&w)[4]) {
  constexpr uint32_t kMag = 0x7FFF7FFFu;
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = __vmaxu2(__vmaxu2(w[i].x & kMag, w[i].y & kMag), __vmaxu2(w[i].z & kMag, w[i].w & kMag));
  const uint32_t c = __vmaxu2(__vmaxu2(p[0], p[1]), __vmaxu2(p[2], p[3]));
  return max(c & 0xFFFFu, c >> 16);
}

// Unbiased block exponent ub from the bf16 magnitude pattern of amax.
__device__ __forceinline__ int block_exponent(uint32_t amax_bits) {
  uint32_t u = ((amax_bits << 16) + 0x200000u) & 0xFF800000u;
  int ub = (int)((u >> 23) & 0xFFu) - 129;
  return min(max(ub, -127), 127);
}

// 2^-ub as an fp32 (ub <= 126 for any bf16 input, so this is a normal number).
__device__ __forceinline__ float inverse_scale(int ub) {
  return __uint_as_float((uint32_t)(127 - ub) << 23);
}

// Magnitude code of a non-negative q by comparison with the grid midpoints;
// a midpoint goes to the neighbour whose code is even.
__device__ __forceinline__ uint32_t e2m1_code_sw(float q) {
  return (uint32_t)(q > 0.25f) + (uint32_t)(q >= 0.75f) + (uint32_t)(q > 1.25f) + (uint32_t)(q >= 1.75f) +
         (uint32_t)(q > 2.5f) + (uint32_t)(q >= 3.5f) + (uint32_t)(q > 5.0f);
}

// Two values -> one byte (lo in bits 0-3, hi in bits 4-7) with the hardware
// round-to-nearest-even, saturating e2m1 conversion.  The first source
// operand of the conversion lands in the upper nibble.
__device__ __forceinline__ uint32_t e2m1x2_hw(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Encode 8 consecutive bf16 values (K order: w.x low half first) with the
// block's inverse scale into 4 bytes of packed e2m1 (byte i holds elements
// 2i and 2i+1).  Values that round to zero keep their sign (0x8 for
// negatives): the hardware conversion does so itself (on GB300 it gives 0x8
// for a negative input that rounds to zero; the GPU tests check every bf16
// value under every block exponent), the comparison encoder takes the signs
// from the inputs.
template <bool kHardwareCvt>
__device__ __forceinline__ uint32_t encode8(const uint4& w, float inv_scale) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = words[i];
    const float x0 = __uint_as_float(v << 16) * inv_scale;
    const float x1 = __uint_as_float(v & 0xFFFF0000u) * inv_scale;
    uint32_t byte;
    if constexpr (kHardwareCvt) {
      byte = e2m1x2_hw(x0, x1) & 0xFFu;
    } else {
      byte = e2m1_code_sw(fabsf(x0)) | (e2m1_code_sw(fabsf(x1)) << 4);
      byte |= ((v >> 12) & 0x8u) | ((v >> 24) & 0x80u);  // input signs -> bits 3 and 7
    }
    out |= byte << (8 * i);
  }
  return out;
}

// One 32-element block (64 bytes of bf16 in K order) -> 16 bytes of packed
// e2m1 (byte i holds elements 2i and 2i+1) and its e8m0 scale byte.  One
// thread owns the whole block, so the block maximum needs no shuffles.
template <bool kHardwareCvt>
__device__ __forceinline__ uint4 quantize_block32(const uint4 (&w)[4], uint32_t& scale_byte) {
  const int ub = block_exponent(absmax32_bits(w));
  scale_byte = (uint32_t)(ub + 127);
  const float inv = inverse_scale(ub);
  return make_uint4(encode8<kHardwareCvt>(w[0], inv), encode8<kHardwareCvt>(w[1], inv),
                    encode8<kHardwareCvt>(w[2], inv), encode8<kHardwareCvt>(w[3], inv));
}

// One 32-element block held by a quad of lanes (lanes 4j..4j+3, 8 bf16 each
// in K order, lane 4j first): the same block maximum, scale and codes as
// quantize_block32, with the maximum reduced across the quad by shuffles.
// Returns this lane's 4 packed bytes (bytes 4q..4q+3 of the block's 16);
// every lane of the quad gets the scale byte.  All 32 lanes must call it.
template <bool kHardwareCvt>
__device__ __forceinline__ uint32_t quantize_quad(const uint4& w, uint32_t& scale_byte) {
  constexpr uint32_t kMag = 0x7FFF7FFFu;
  const uint32_t c = __vmaxu2(__vmaxu2(w.x & kMag, w.y & kMag), __vmaxu2(w.z & kMag, w.w & kMag));
  uint32_t m = max(c & 0xFFFFu, c >> 16);
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  const int ub = block_exponent(m);
  scale_byte = (uint32_t)(ub + 127);
  return encode8<kHardwareCvt>(w, inverse_scale(ub));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The 64 bytes of one 32-element block from global memory (read-only path).
__device__ __forceinline__ void ldg_nc_block(const uint16_t* p, uint4 (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = ldg_nc_v4(p + 8 * i);
}

// seg / d, in 32-bit arithmetic when every segment index involved fits
// (a 64-bit division is a long software sequence on the GPU).
__device__ __forceinline__ int64_t div_seg(int64_t seg, int64_t d, bool small) {
  return small ? (int64_t)((uint32_t)seg / (uint32_t)d) : seg / d;
}

// Activation image writer, one warp per row segment: 256 consecutive K
// elements (8 scale blocks) of one row.  Lane l holds elements 8l..8l+7 (one
// 16-byte load; the warp reads 512 contiguous bytes), a quad of lanes holds
// one block and reduces its maximum by shuffles; the warp's 32 four-byte
// stores fill one swizzled 128-byte row of a data tile and two lanes store
// the row's scale words (blocks 0-3 and 4-7).  Segment s is row s / kt_count,
// K block s % kt_count.  The calling warp takes segments lo + first,
// lo + first + stride, ... below hi, in batches of kBatch, software-pipelined:
// the loads of the next batch are issued before the current batch is
// quantized, so a warp's memory latency overlaps its own arithmetic.  Each
// step moves the row and K block by the same amounts, so they are advanced
// incrementally instead of divided out per segment.  Rows >= m and K beyond
// k are written as zero codes with scale byte 0.  All 32 lanes must call it.
template <bool kHw, int kBatch>
__device__ __forceinline__ void quantize_image_segments(const uint16_t* __restrict__ a, int64_t m, int64_t k,
                                                        int64_t lda, uint8_t* __restrict__ img, int64_t kt_count,
                                                        int64_t lo, int64_t hi, int64_t first, int64_t stride,
                                                        int lane) {
  int64_t seg = lo + first;
  if (seg >= hi) return;
  int64_t row = seg / kt_count, kt = seg - row * kt_count;
  const int64_t d_row = stride / kt_count, d_kt = stride - d_row * kt_count;
  const int b = lane >> 2;
  auto load = [&](int64_t r, int64_t t, bool ok) -> uint4 {
    const int64_t col = t * kTileK + lane * 8;
    return (ok && r < m && col < k) ? ldg_nc_v4(a + r * lda + col) : make_uint4(0, 0, 0, 0);
  };
  // the next segment of this warp: its row, K block, validity and bf16 data
  auto take = [&](int64_t& r_out, int64_t& kt_out, bool& ok_out, uint4& v_out) {
    r_out = row;
    kt_out = kt;
    ok_out = seg < hi;
    v_out = load(row, kt, ok_out);
    seg += stride;
    row += d_row;
    kt += d_kt;
    if (kt >= kt_count) {
      kt -= kt_count;
      ++row;
    }
  };
  uint4 cur[kBatch];
  int64_t crow[kBatch], ckt[kBatch];
  bool cval[kBatch];
#pragma unroll
  for (int i = 0; i < kBatch; ++i) take(crow[i], ckt[i], cval[i], cur[i]);
  while (cval[0]) {
    uint4 nxt[kBatch];
    int64_t nrow[kBatch], nkt[kBatch];
    bool nval[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) take(nrow[i], nkt[i], nval[i], nxt[i]);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (!cval[i]) break;  // uniform across the warp
      uint32_t sbyte;
      const uint32_t packed = quantize_quad<kHw>(cur[i], sbyte);
      const int r = (int)(crow[i] & (kTileRows - 1));
      uint8_t* tile = img + image_block(crow[i] / kTileRows, ckt[i], kt_count);
      *reinterpret_cast<uint32_t*>(tile + tile_data_offset(r, b * 16 + (lane & 3) * 4)) = packed;
      // scale word of blocks 0-3 (atom 0) and of blocks 4-7 (atom 1): byte b & 3
      uint32_t word = sbyte << (8 * (b & 3));
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 4);
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 8);
      if ((lane & 15) == 0) *reinterpret_cast<uint32_t*>(tile + kTileDataBytes + tile_sf_offset(r, b)) = word;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      cur[i] = nxt[i];
      crow[i] = nrow[i];
      ckt[i] = nkt[i];
      cval[i] = nval[i];
    }
  }
}

}  // namespace mxfp4
