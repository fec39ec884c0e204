// MXFP4 quantization and weight-prepack kernels (HBM-bound; no tensor cores).
//
//   quant_linear_kernel : bf16 A[m,k] -> packed e2m1 [m,k/2] + e8m0 [m,k/32]
//   quant_image_kernel  : bf16 A[m,k] -> tiled operand image (see mxfp4_device.cuh)
//   prepack_*_kernel    : linear MXFP4 B -> tiled operand image
//
// One thread owns one 32-element scale block: it loads the block's 64 bytes,
// forms the block maximum in registers and writes 16 packed bytes plus the
// scale byte.  Consecutive threads take consecutive blocks of a row, so a
// warp reads 2 KiB of contiguous bf16 and writes 512 contiguous bytes.
#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_launch.h"
#include "ptx.cuh"

namespace mxfp4 {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;  // blocks in flight per thread

template <bool kHw>
__global__ void __launch_bounds__(kQuantThreads)
    quant_linear_kernel(const uint16_t* __restrict__ a, int64_t m, int64_t k, int64_t lda,
                        uint8_t* __restrict__ q, uint8_t* __restrict__ scale) {
  const int64_t blocks_per_row = k / 32;
  const int64_t total = m * blocks_per_row;
  const int64_t nthreads = (int64_t)gridDim.x * kQuantThreads;
  const int64_t t0 = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x;
  for (int64_t base = t0; base < total; base += nthreads * kQuantUnroll) {
    uint4 w[kQuantUnroll][4];
    int64_t row[kQuantUnroll], blk[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t t = base + (int64_t)u * nthreads;
      row[u] = t / blocks_per_row;
      blk[u] = t - row[u] * blocks_per_row;
      if (t < total) ldg_nc_block(a + row[u] * lda + blk[u] * 32, w[u]);
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      if (base + (int64_t)u * nthreads >= total) continue;
      uint32_t sbyte;
      const uint4 packed = quantize_block32<kHw>(w[u], sbyte);
      *reinterpret_cast<uint4*>(q + row[u] * (k / 2) + blk[u] * 16) = packed;
      scale[row[u] * blocks_per_row + blk[u]] = (uint8_t)sbyte;
    }
  }
}

// Writes the operand image of an m-row matrix: rows [0, rows_out) of the
// image, rows >= m as zeros (rows_out = m leaves the last row tile's padding
// rows untouched: an activation's padding rows only reach accumulator rows
// that are never stored; a weight image needs them zero).  K beyond k up to
// the tile edge is written as zeros.  Thread t covers block b = t % 8 of K
// block kt of a row, so eight consecutive threads write one swizzled
// 128-byte row of a data tile.
template <bool kHw>
__global__ void __launch_bounds__(kQuantThreads)
    quant_image_kernel(const uint16_t* __restrict__ a, int64_t m, int64_t k, int64_t lda,
                       uint8_t* __restrict__ img, int64_t rows_out) {
  // Let the dependent GEMM launch now: it prefetches weights and waits for
  // this grid's completion before it reads the image.
  pdl_launch_dependents();
  const int64_t kt_count = ceil_div(k, kTileK);
  const int64_t total = rows_out * kt_count * 8;
  const int64_t nthreads = (int64_t)gridDim.x * kQuantThreads;
  const int64_t t0 = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x;
  for (int64_t base = t0; base < total; base += nthreads * kQuantUnroll) {
    uint4 w[kQuantUnroll][4];
    int64_t row[kQuantUnroll], kt[kQuantUnroll];
    int b[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t t = base + (int64_t)u * nthreads;
      b[u] = (int)(t & 7);
      row[u] = (t >> 3) / kt_count;
      kt[u] = (t >> 3) - row[u] * kt_count;
      const int64_t col = kt[u] * kTileK + b[u] * 32;
      if (t < total && col < k && row[u] < m) {
        ldg_nc_block(a + row[u] * lda + col, w[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[u][i] = make_uint4(0, 0, 0, 0);  // padding: zero codes, scale byte 0
      }
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      if (base + (int64_t)u * nthreads >= total) continue;
      uint32_t sbyte;
      const uint4 packed = quantize_block32<kHw>(w[u], sbyte);
      const int r = (int)(row[u] & (kTileRows - 1));
      uint8_t* tile = img + image_block(row[u] / kTileRows, kt[u], kt_count);
      *reinterpret_cast<uint4*>(tile + tile_data_offset(r, b[u] * 16)) = packed;
      tile[kTileDataBytes + tile_sf_offset(r, b[u])] = (uint8_t)sbyte;
    }
  }
}

// Linear MXFP4 B (q [n,k/2], scale [n,k/32]) -> tiled image; one thread per
// 16-byte data chunk or per scale byte.  Padding rows and K are zero.
__global__ void __launch_bounds__(256)
    prepack_data_kernel(const uint8_t* __restrict__ bq, int64_t n, int64_t k, uint8_t* __restrict__ img) {
  const int64_t kt_count = ceil_div(k, kTileK);
  const int64_t total = ceil_div(n, kTileRows) * kt_count * (kTileDataBytes / 16);
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = idx / (kTileDataBytes / 16);
    const int within = (int)(idx % (kTileDataBytes / 16));
    const int r = within >> 3, c = within & 7;
    const int64_t row = (tile / kt_count) * kTileRows + r;
    const int64_t kbyte = (tile % kt_count) * (kTileK / 2) + c * 16;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < n && kbyte < k / 2) v = *reinterpret_cast<const uint4*>(bq + row * (k / 2) + kbyte);
    *reinterpret_cast<uint4*>(img + tile * kTileBytes + tile_data_offset(r, c * 16)) = v;
  }
}

__global__ void __launch_bounds__(256)
    prepack_scale_kernel(const uint8_t* __restrict__ bs, int64_t n, int64_t k, uint8_t* __restrict__ img) {
  const int64_t kt_count = ceil_div(k, kTileK);
  const int64_t total = ceil_div(n, kTileRows) * kt_count * kTileSfBytes;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = idx / kTileSfBytes;
    const int within = (int)(idx % kTileSfBytes);
    const int r = within >> 3, b = within & 7;
    const int64_t row = (tile / kt_count) * kTileRows + r;
    const int64_t blk = (tile % kt_count) * (kTileK / 32) + b;
    uint8_t v = 0;
    if (row < n && blk < k / 32) v = bs[row * (k / 32) + blk];
    img[tile * kTileBytes + kTileDataBytes + tile_sf_offset(r, b)] = v;
  }
}

// ------------------------------------------------------------ launchers
static int grid_for(int64_t work_items, int per_block) {
  int sms = num_sms();
  int64_t blocks = ceil_div(work_items, per_block);
  int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

cudaError_t launch_quant_linear(const void* a, int64_t m, int64_t k, int64_t lda, void* q, void* scale,
                                cudaStream_t stream) {
  const int grid = grid_for(m * (k / 32), kQuantThreads);
  quant_linear_kernel<kUseHardwareCvt><<<grid, kQuantThreads, 0, stream>>>(
      static_cast<const uint16_t*>(a), m, k, lda, static_cast<uint8_t*>(q), static_cast<uint8_t*>(scale));
  return cudaGetLastError();
}

cudaError_t launch_quant_image(const void* a, int64_t m, int64_t k, int64_t lda, void* img, cudaStream_t stream,
                               bool zero_padding_rows) {
  const int64_t rows_out = zero_padding_rows ? ceil_div(m, kTileRows) * kTileRows : m;
  const int grid = grid_for(rows_out * ceil_div(k, kTileK) * 8, kQuantThreads);
  quant_image_kernel<kUseHardwareCvt><<<grid, kQuantThreads, 0, stream>>>(
      static_cast<const uint16_t*>(a), m, k, lda, static_cast<uint8_t*>(img), rows_out);
  return cudaGetLastError();
}

cudaError_t launch_prepack(const void* bq, const void* bs, int64_t n, int64_t k, void* img, cudaStream_t stream) {
  const int64_t tiles = ceil_div(n, kTileRows) * ceil_div(k, kTileK);
  prepack_data_kernel<<<grid_for(tiles * (kTileDataBytes / 16), 256), 256, 0, stream>>>(
      static_cast<const uint8_t*>(bq), n, k, static_cast<uint8_t*>(img));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prepack_scale_kernel<<<grid_for(tiles * kTileSfBytes, 256), 256, 0, stream>>>(
      static_cast<const uint8_t*>(bs), n, k, static_cast<uint8_t*>(img));
  return cudaGetLastError();
}

}  // namespace mxfp4
