// MXFP4 quantization and weight-prepack kernels (HBM-bound; no tensor cores).
//
//   quant_linear_kernel : bf16 A[m,k] -> packed e2m1 [m,k/2] + e8m0 [m,k/32]
//   quant_image_kernel  : bf16 A[m,k] -> tiled operand image (see mxfp4_device.cuh)
//   prepack_*_kernel    : linear MXFP4 B -> tiled operand image
//
// A warp quantizes 256-element row segments (four lanes per 32-element
// block), reading 512 contiguous bytes per load instruction.
#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_launch.h"
#include "ptx.cuh"

namespace mxfp4 {

constexpr int kQuantThreads = 256;
constexpr int kQuantSegBatch = 4;  // row segments whose loads one warp keeps in flight
constexpr int kImageSegBatch = 2;  // the image writer's batch (two batches in registers)

// Both quantizers work in row segments: 256 consecutive K elements (8 scale
// blocks) of one row, one segment per warp.  Lane l holds elements 8l..8l+7
// (one 16-byte load; the warp reads 512 contiguous bytes), a quad of lanes
// holds one block, and the block maximum is reduced across the quad.  A warp
// loads up to kQuantSegBatch segments before quantizing any, so enough bytes
// are in flight to cover HBM latency with few registers per thread.
// Segments are dealt round-robin over all warps of the grid.

// bf16 A[m,k] -> packed e2m1 [m,k/2] + e8m0 [m,k/32] (k a multiple of 32).
template <bool kHw>
__global__ void __launch_bounds__(kQuantThreads)
    quant_linear_kernel(const uint16_t* __restrict__ a, int64_t m, int64_t k, int64_t lda,
                        uint8_t* __restrict__ q, uint8_t* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t segs_per_row = ceil_div(k, kTileK);
  const int64_t total = m * segs_per_row;
  const bool small = total + (int64_t)gridDim.x * kQuantThreads * kQuantSegBatch < (1ll << 31);
  const int64_t warps = (int64_t)gridDim.x * (kQuantThreads / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
  for (int64_t base = w0; base < total; base += warps * kQuantSegBatch) {
    uint4 v[kQuantSegBatch];
    int64_t row[kQuantSegBatch], col[kQuantSegBatch];
#pragma unroll
    for (int i = 0; i < kQuantSegBatch; ++i) {
      const int64_t seg = base + (int64_t)i * warps;
      row[i] = div_seg(seg, segs_per_row, small);
      col[i] = (seg - row[i] * segs_per_row) * kTileK + lane * 8;
      v[i] = (seg < total && col[i] < k) ? ldg_nc_v4(a + row[i] * lda + col[i]) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kQuantSegBatch; ++i) {
      if (base + (int64_t)i * warps >= total) break;  // uniform across the warp
      uint32_t sbyte;
      const uint32_t packed = quantize_quad<kHw>(v[i], sbyte);
      if (col[i] < k) {
        *reinterpret_cast<uint32_t*>(q + row[i] * (k / 2) + col[i] / 2) = packed;
        if ((lane & 3) == 0) scale[row[i] * (k / 32) + col[i] / 32] = (uint8_t)sbyte;
      }
    }
  }
}

// Writes the operand image of an m-row matrix: rows [0, rows_out) of the
// image, rows >= m as zeros (rows_out = m leaves the last row tile's padding
// rows untouched: an activation's padding rows only reach accumulator rows
// that are never stored; a weight image needs them zero).  K beyond k up to
// the tile edge is written as zeros.  Segments are dealt round-robin over
// every warp of the grid (quantize_image_segments).
template <bool kHw>
__global__ void __launch_bounds__(kQuantThreads)
    quant_image_kernel(const uint16_t* __restrict__ a, int64_t m, int64_t k, int64_t lda,
                       uint8_t* __restrict__ img, int64_t rows_out) {
  // Let the dependent GEMM launch now: it prefetches weights and waits for
  // this grid's completion before it reads the image.
  pdl_launch_dependents();
  const int64_t kt_count = ceil_div(k, kTileK);
  const int64_t warps = (int64_t)gridDim.x * (kQuantThreads / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
  quantize_image_segments<kHw, kImageSegBatch>(a, m, k, lda, img, kt_count, 0, rows_out * kt_count, w0, warps,
                                               threadIdx.x & 31);
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

// Grid of the quantization kernels: one warp per segment, up to `per_sm`
// 256-thread CTAs per SM; beyond that each warp takes several segments.
// The weight quantizer runs up to eight CTAs per SM (about two resident
// waves at its register count), loading kQuantSegBatch segments at a time.
// The activation image writer runs one resident wave (four CTAs per SM at
// its 64 registers) whose warps pipeline their segments: measured on GB300
// at m = 4096, k = 2048 the quantizer alone takes the same time either way
// (it reads A at what DRAM gives after an L2 flush by writes), but the
// dependent GEMM's call finished 1.0 us sooner with the single wave.
static int quant_grid(int64_t segments, int per_sm) {
  const int64_t max_warps = (int64_t)num_sms() * per_sm * (kQuantThreads / 32);
  const int64_t warps = segments < max_warps ? segments : max_warps;
  const int64_t blocks = ceil_div(warps, (int64_t)(kQuantThreads / 32));
  return blocks < 1 ? 1 : (int)blocks;
}

cudaError_t launch_quant_linear(const void* a, int64_t m, int64_t k, int64_t lda, void* q, void* scale,
                                cudaStream_t stream) {
  const int grid = quant_grid(m * ceil_div(k, kTileK), 8);
  quant_linear_kernel<kUseHardwareCvt><<<grid, kQuantThreads, 0, stream>>>(
      static_cast<const uint16_t*>(a), m, k, lda, static_cast<uint8_t*>(q), static_cast<uint8_t*>(scale));
  return cudaGetLastError();
}

cudaError_t launch_quant_image(const void* a, int64_t m, int64_t k, int64_t lda, void* img, cudaStream_t stream,
                               bool zero_padding_rows) {
  const int64_t rows_out = zero_padding_rows ? ceil_div(m, kTileRows) * kTileRows : m;
  const int grid = quant_grid(rows_out * ceil_div(k, kTileK), 4);
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
