// mxfp4_gemm_noalloc: mxfp4_gemm for callers that cannot provide workspace.
//
// Some callers cannot allocate device memory or pass a workspace through:
// a plugin whose host framework's call signature has no scratch argument,
// or an engine whose memory planner has already committed every byte of
// device memory before the first call.  For them this entry point keeps the
// scratch it needs (the tiled operand image of A when m > 32) in a
// file-scope device array that is part of the library's image, so it
// allocates nothing when called.
//
// Cost and limits: every device that loads the library holds the array
// (kNoallocScratchBytes) until the process exits.  Shapes whose scratch need
// is larger are rejected before anything is enqueued.  All calls on a
// device share the one array, so calls that overlap on the GPU (different
// streams, no ordering between them) race on it; calls in one stream are
// ordered and safe.  The scratch is fully rewritten by every call that uses
// it, so nothing in it has to start at zero.
#include <cuda_runtime.h>

#include <atomic>

#include "mxfp4.h"
#include "mxfp4_device.cuh"
#include "mxfp4_launch.h"

namespace {

constexpr size_t kNoallocScratchBytes = MXFP4_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch[kMaxDevices];

// Device address of the scratch array on the current device, looked up while
// that device is current.  (In host code the array's name only stands for the
// symbol; it is never a usable device pointer.)  Only a successful lookup is
// kept: a lookup that failed (say, one made during a stream capture) is tried
// again by the next call.  Two threads that miss at once both look it up and
// store the same address.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      (void)cudaGetLastError();  // not sticky: the next call tries again
      return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    }
    g_scratch[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" MXFP4_API mxfp4_status mxfp4_gemm_noalloc(const void* a_bf16, int64_t m, int64_t k, int64_t lda,
                                                      const void* b_packed, int64_t n, void* c_bf16, int64_t ldc,
                                                      void* stream) {
  if (m <= 0 || n <= 0 || k <= 0 || (k % 32) != 0 || lda < k || (lda % 8) != 0 || ldc < n || (ldc % 8) != 0)
    return MXFP4_ERR_INVALID_ARG;
  if (!a_bf16 || !b_packed || !c_bf16 || !aligned16(a_bf16) || !aligned16(b_packed) || !aligned16(c_bf16))
    return MXFP4_ERR_INVALID_ARG;
  mxfp4::GemmPlan plan;
  if (mxfp4::make_gemm_plan(m, n, k, &plan) != 0) return MXFP4_ERR_UNSUPPORTED;
  if (plan.workspace > kNoallocScratchBytes) return MXFP4_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (plan.workspace > 0 && scratch_on_current_device(&scratch) != cudaSuccess) return MXFP4_ERR_CUDA;
  const cudaError_t e = mxfp4::launch_gemm(plan, a_bf16, m, k, lda, b_packed, n, c_bf16, ldc, scratch,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}
