// Dense FP4 tensor-core rate of this GPU: the denominator of the large-m
// GEMM's roofline fraction (the measured peak figures at hand cover HBM
// and bf16 only).  One CTA per SM keeps a 128 x 256 fp32 accumulator in
// tensor memory and one thread issues back-to-back 128 x 256 x 256
// block-scaled K blocks (tcgen05.mma kind::mxf4, eight MMAs of 128 x 128 x 64
// per block, the GEMM kernels' own issue sequence) on operands that stay in
// shared memory; nothing is loaded from or stored to global memory.  The
// host times the launch with CUDA events and divides the FLOPs by it.  Also
// the launch floors: empty kernels, and minimal kernels that touch global
// and tensor memory, timed the way the GEMMs are.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "mxfp4.h"
#include "mxfp4_launch.h"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int kPeakThreads = 128;
constexpr int kOperandBytes = 3 * 16384;  // A (128 rows x 256 K) and two 128-row B halves, e2m1
// More than half of an SM's shared memory, so that exactly one CTA (and one
// 512-column tensor-memory allocation) is resident per SM.
constexpr int kPeakSmemBytes = 120 * 1024;
constexpr long long kPeakWaitCycles = 1ll << 34;  // ~8 s at 2 GHz: far beyond any valid launch

__device__ int g_peak_timeout = 0;

__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int64_t kblocks) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Operands: a hashed bit pattern (every e2m1 code occurs); the layout
  // descriptors are those of the GEMM's swizzled tiles.
  for (int i = threadIdx.x; i < kOperandBytes / 4; i += kPeakThreads) {
    uint32_t v = (uint32_t)i * 2654435761u;
    v ^= v >> 15;
    reinterpret_cast<uint32_t*>(smem)[i] = v;
  }
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();  // the operand bytes are read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // Scale factors (e8m0 127 = 2^0) for A and both B halves in columns
  // 256-279 of every lane: warp w writes quadrant w.
  {
    const uint32_t ones[8] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu,
                              0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
    const uint32_t base = tmem + ((uint32_t)(warp * 32) << 16) + 256;
    tmem_store_8(base, ones);
    tmem_store_8(base + 8, ones);
    tmem_store_8(base + 16, ones);
    tmem_store_wait();
  }
  (void)lane;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    const uint64_t ad = smem_desc(smem_addr(smem), 0, 1024, kLayoutSwizzle128);
    const uint64_t bd0 = smem_desc(smem_addr(smem + 16384), 0, 1024, kLayoutSwizzle128);
    const uint64_t bd1 = smem_desc(smem_addr(smem + 32768), 0, 1024, kLayoutSwizzle128);
    const uint32_t ie = idesc_mxf4(128, 128, 0, 0), io = idesc_mxf4(128, 128, 2, 2);
    for (int64_t it = 0; it < kblocks; ++it)
      mma_mxf4_kblock_n256(tmem, ad, bd0, bd1, ie, io, tmem + 256, tmem + 264, tmem + 272, it > 0 ? 1u : 0u);
    mma_commit(&done);  // fires when every MMA above has completed
    const long long t0 = clock64();
    while (!mbar_try_wait(&done, 0)) {
      if (clock64() - t0 > kPeakWaitCycles) {  // not expected: report it and stop waiting
        atomicExch(&g_peak_timeout, 1);
        break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// An empty kernel: the launch floor that the small-m GEMM's time is read against.
__global__ void empty_kernel() {}

// The least a GEMM launch does: read a word of global memory, allocate and
// free tensor memory, write a word.  After an L2 flush by writes, each of the
// three alone already costs a kernel about 2 us of event time over the empty
// one (measured on GB300), so this is the floor a tcgen05 GEMM meets.
__device__ uint32_t g_minimal_words[4096 * 2];
__global__ void minimal_kernel() {
  __shared__ uint32_t slot;
  const int i = blockIdx.x & 4095;
  uint32_t v = 0;
  if (threadIdx.x == 0) v = *reinterpret_cast<volatile uint32_t*>(&g_minimal_words[2 * i]);
  tmem_alloc(&slot, 32);
  tmem_relinquish();
  tc_fence_before();
  __syncwarp();
  tc_fence_after();
  tmem_dealloc(slot, 32);
  if (threadIdx.x == 0) g_minimal_words[2 * i + 1] = v + 1;
}

}  // namespace
}  // namespace mxfp4

extern "C" mxfp4_status mxfp4_launch_empty(int count, int ctas, void* stream) {
  if (count < 1 || count > 16 || ctas < 1 || ctas > 65535) return MXFP4_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    mxfp4::empty_kernel<<<ctas, 32, 0, static_cast<cudaStream_t>(stream)>>>();
    if (cudaGetLastError() != cudaSuccess) return MXFP4_ERR_CUDA;
  }
  return MXFP4_OK;
}

extern "C" mxfp4_status mxfp4_launch_minimal(int count, int ctas, void* stream) {
  if (count < 1 || count > 16 || ctas < 1 || ctas > 65535) return MXFP4_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    mxfp4::minimal_kernel<<<ctas, 32, 0, static_cast<cudaStream_t>(stream)>>>();
    if (cudaGetLastError() != cudaSuccess) return MXFP4_ERR_CUDA;
  }
  return MXFP4_OK;
}

extern "C" mxfp4_status mxfp4_measure_fp4_peak(int64_t kblocks_per_sm, double* tflops, void* stream) {
  using namespace mxfp4;
  if (kblocks_per_sm <= 0 || kblocks_per_sm > (int64_t(1) << 24) || !tflops) return MXFP4_ERR_INVALID_ARG;
  static std::atomic<bool> attr_done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXFP4_ERR_CUDA;
  if (dev >= 0 && dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmemBytes) !=
        cudaSuccess)
      return MXFP4_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  const int sms = num_sms();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return MXFP4_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return MXFP4_ERR_CUDA;
  }
  mxfp4_status status = MXFP4_OK;
  int timed_out = 0;
  float ms = 0.f;
  if (cudaEventRecord(e0, st) != cudaSuccess) status = MXFP4_ERR_CUDA;
  if (status == MXFP4_OK) {
    mma_peak_kernel<<<sms, kPeakThreads, kPeakSmemBytes, st>>>(kblocks_per_sm);
    if (cudaGetLastError() != cudaSuccess) status = MXFP4_ERR_CUDA;
  }
  if (status == MXFP4_OK && (cudaEventRecord(e1, st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                             cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
    status = MXFP4_ERR_CUDA;
  if (status == MXFP4_OK) {
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&timed_out, g_peak_timeout, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_peak_timeout, &zero, sizeof(int)) != cudaSuccess)
      status = MXFP4_ERR_CUDA;
    else if (timed_out)
      status = MXFP4_ERR_TIMEOUT;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (status != MXFP4_OK) return status;
  // 2 * 128 * 256 * 256 FLOPs per K block per SM
  const double flops = 2.0 * 128 * 256 * 256 * (double)kblocks_per_sm * sms;
  *tflops = ms > 0.f ? flops / (ms * 1e-3) / 1e12 : 0.0;
  return MXFP4_OK;
}
