// MXFP4 quantization and weight-prepack kernels (HBM-bound; no tensor cores).
//
//   quant_linear_kernel : bf16 A[m,k] -> packed e2m1 [m,k/2] + e8m0 [m,k/32]
//   quant_image_kernel  : bf16 A[m,k] -> tiled operand image (see mxfp4_device.cuh)
//   prepack_*_kernel    : linear MXFP4 B -> tiled operand image
//
// One warp covers 256 consecutive K elements of one row: lane l loads 16
// bytes (8 bf16), lanes 4j..4j+3 form 32-element block j, the block maximum
// comes from two shuffles, and each lane writes 4 packed bytes.
#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_launch.h"
#include "ptx.cuh"

namespace mxfp4 {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;

template <bool kHw>
__global__ void __launch_bounds__(kQuantThreads)
    quant_linear_kernel(const uint16_t* __restrict__ a, int64_t m, int64_t k, int64_t lda,
                        uint8_t* __restrict__ q, uint8_t* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t spans_per_row = ceil_div(k, kTileK);
  const int64_t total = m * spans_per_row;
  const int64_t nwarps = (int64_t)gridDim.x * (kQuantThreads / 32);
  const int64_t warp0 = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
  const int64_t qstride = k / 2, sstride = k / 32;
  for (int64_t base = warp0; base < total; base += nwarps * kQuantUnroll) {
    uint4 w[kQuantUnroll];
    int64_t row[kQuantUnroll], col[kQuantUnroll];
    bool ok[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t t = base + (int64_t)u * nwarps;
      row[u] = t / spans_per_row;
      col[u] = (t - row[u] * spans_per_row) * kTileK + lane * 8;
      ok[u] = (t < total) && (col[u] < k);
      w[u] = ok[u] ? ldg_nc_v4(a + row[u] * lda + col[u]) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      uint32_t sbyte;
      const uint32_t packed = quantize_lane<kHw>(w[u], sbyte);
      if (ok[u]) {
        *reinterpret_cast<uint32_t*>(q + row[u] * qstride + col[u] / 2) = packed;
        if ((lane & 3) == 0) scale[row[u] * sstride + col[u] / 32] = (uint8_t)sbyte;
      }
    }
  }
}

// Writes the A-side operand image of an m-row activation for the GEMM.
// Rows >= m of the last row tile are left untouched (their accumulator rows
// are never stored); K beyond k up to the tile edge is written as zeros.
template <bool kHw>
__global__ void __launch_bounds__(kQuantThreads)
    quant_image_kernel(const uint16_t* __restrict__ a, int64_t m, int64_t k, int64_t lda,
                       uint8_t* __restrict__ img) {
  // Let the dependent GEMM launch now: it prefetches weights and waits for
  // this grid's completion before it reads the image.
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t kt_count = ceil_div(k, kTileK);
  const int64_t total = m * kt_count;
  const int64_t nwarps = (int64_t)gridDim.x * (kQuantThreads / 32);
  const int64_t warp0 = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
  for (int64_t base = warp0; base < total; base += nwarps * kQuantUnroll) {
    uint4 w[kQuantUnroll];
    int64_t row[kQuantUnroll], kt[kQuantUnroll];
    bool live[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t t = base + (int64_t)u * nwarps;
      live[u] = t < total;
      row[u] = t / kt_count;
      kt[u] = t - row[u] * kt_count;
      const int64_t col = kt[u] * kTileK + lane * 8;
      w[u] = (live[u] && col < k) ? ldg_nc_v4(a + row[u] * lda + col) : make_uint4(0, 0, 0, 0);
    }
    // all-zero pieces quantize to zero nibbles and scale byte 0
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      uint32_t sbyte;
      const uint32_t packed = quantize_lane<kHw>(w[u], sbyte);
      if (live[u]) {
        const int r = (int)(row[u] & (kTileRows - 1));
        uint8_t* blk = img + image_block(row[u] / kTileRows, kt[u], kt_count);
        *reinterpret_cast<uint32_t*>(blk + tile_data_offset(r, lane * 4)) = packed;
        if ((lane & 3) == 0) blk[kTileDataBytes + tile_sf_offset(r, lane >> 2)] = (uint8_t)sbyte;
      }
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
  const int64_t warps = m * ceil_div(k, kTileK);
  const int grid = grid_for(warps, (kQuantThreads / 32) * kQuantUnroll);
  quant_linear_kernel<kUseHardwareCvt><<<grid, kQuantThreads, 0, stream>>>(
      static_cast<const uint16_t*>(a), m, k, lda, static_cast<uint8_t*>(q), static_cast<uint8_t*>(scale));
  return cudaGetLastError();
}

cudaError_t launch_quant_image(const void* a, int64_t m, int64_t k, int64_t lda, void* img, cudaStream_t stream) {
  const int64_t warps = m * ceil_div(k, kTileK);
  const int grid = grid_for(warps, (kQuantThreads / 32) * kQuantUnroll);
  quant_image_kernel<kUseHardwareCvt><<<grid, kQuantThreads, 0, stream>>>(static_cast<const uint16_t*>(a), m, k,
                                                                          lda, static_cast<uint8_t*>(img));
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
