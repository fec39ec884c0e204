// C ABI of the MXFP4 library: argument validation, then kernel launches on
// the caller's stream.  Nothing here allocates device memory or blocks,
// except mxfp4_device_status; mxfp4_gemm_host keeps one helper stream and a
// few events per host thread and device for its chunked round trip.
#include <cuda_runtime.h>

#include <cstdint>

#include "mxfp4.h"
#include "mxfp4_device.cuh"
#include "mxfp4_launch.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mxfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA; }

bool valid_k(int64_t k) { return k > 0 && (k % 32) == 0; }

// The address through which kernels reach page-locked host memory (mapped
// into every device's address space under unified addressing), else nullptr
// (pageable memory, or a pointer the runtime does not know).
// Largest k for which mxfp4_gemm_host lets the fused kernel work on host
// memory directly.
constexpr int64_t kDirectHostMaxK = 512;

// Round trips whose C is at least kChunkMinCBytes split m into up to
// kMaxChunks row chunks of whole 256-row tiles: each chunk's C goes down on a
// helper stream while the next chunk's A goes up and its GEMM runs on the
// caller's stream.  The host link carries both directions at once (on GB300
// ~190-205 GB/s each way; a 58.7 MB download took 311 us alone and 327 us
// beside an upload), so at m = 4096, n = 7168 the downloads of the first
// chunks hide the rest of the work: 437 us in one stream, 378 us in four
// chunks, 409 us in eight (more, smaller GEMMs and copies).
constexpr size_t kChunkMinCBytes = size_t(8) << 20;
constexpr int kMaxChunks = 4;
constexpr int64_t kChunkRowAlign = 256;

// The helper stream and events of the calling host thread on the current
// device, created on first use and kept for the life of the thread (they
// are never destroyed); nullptr if they do not exist and may not be created
// now (during stream capture), or if creating them failed, in which case
// the caller takes the single-stream path.
struct HostPipe {
  cudaStream_t stream = nullptr;
  cudaEvent_t ev[kMaxChunks + 1] = {};
  bool ready = false;
  bool failed = false;
};

HostPipe* host_pipe(bool may_create) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return nullptr;
  }
  thread_local HostPipe pipes[64];
  HostPipe& p = pipes[dev];
  if (p.ready) return &p;
  if (p.failed || !may_create) return nullptr;
  bool ok = cudaStreamCreateWithFlags(&p.stream, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i <= kMaxChunks; ++i)
    ok = cudaEventCreateWithFlags(&p.ev[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    (void)cudaGetLastError();
    p.failed = true;
    return nullptr;
  }
  p.ready = true;
  return &p;
}

void* mapped_host(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();  // not sticky: keep it out of the launch checks
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

}  // namespace

extern "C" {

const char* mxfp4_status_string(int status) {
  switch (status) {
    case MXFP4_OK: return "MXFP4_OK";
    case MXFP4_ERR_INVALID_ARG: return "MXFP4_ERR_INVALID_ARG";
    case MXFP4_ERR_UNSUPPORTED: return "MXFP4_ERR_UNSUPPORTED";
    case MXFP4_ERR_WORKSPACE: return "MXFP4_ERR_WORKSPACE";
    case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA";
    case MXFP4_ERR_TIMEOUT: return "MXFP4_ERR_TIMEOUT";
    default: return "MXFP4_ERR_UNKNOWN";
  }
}

int mxfp4_version(void) { return 100; }

mxfp4_status mxfp4_quant(const void* a_bf16, int64_t m, int64_t k, int64_t lda, void* a_fp4, void* a_scale,
                         void* stream) {
  if (m < 0 || !valid_k(k) || lda < k || (lda % 8) != 0) return MXFP4_ERR_INVALID_ARG;
  if (m == 0) return MXFP4_OK;
  if (!a_bf16 || !a_fp4 || !a_scale || !aligned16(a_bf16) || !aligned16(a_fp4)) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(
      mxfp4::launch_quant_linear(a_bf16, m, k, lda, a_fp4, a_scale, static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_prepacked_b_bytes(int64_t n, int64_t k) {
  if (n <= 0 || !valid_k(k)) return 0;
  return static_cast<size_t>(mxfp4::image_bytes(n, k));
}

mxfp4_status mxfp4_prepack_b(const void* b_fp4, const void* b_scale, int64_t n, int64_t k, void* b_packed,
                             size_t b_packed_bytes, void* stream) {
  if (n <= 0 || !valid_k(k)) return MXFP4_ERR_INVALID_ARG;
  if (!b_fp4 || !b_scale || !b_packed || !aligned16(b_fp4) || !aligned16(b_packed)) return MXFP4_ERR_INVALID_ARG;
  if (b_packed_bytes < mxfp4_prepacked_b_bytes(n, k)) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(mxfp4::launch_prepack(b_fp4, b_scale, n, k, b_packed, static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  mxfp4::GemmPlan plan;
  if (m <= 0 || n <= 0 || !valid_k(k)) return 0;
  if (mxfp4::make_gemm_plan(m, n, k, &plan) != 0) return 0;
  return plan.workspace;
}

mxfp4_status mxfp4_gemm(const void* a_bf16, int64_t m, int64_t k, int64_t lda, const void* b_packed, int64_t n,
                        void* c_bf16, int64_t ldc, void* workspace, size_t workspace_bytes, void* stream) {
  if (m <= 0 || n <= 0 || !valid_k(k) || lda < k || (lda % 8) != 0 || ldc < n || (ldc % 8) != 0)
    return MXFP4_ERR_INVALID_ARG;
  if (!a_bf16 || !b_packed || !c_bf16 || !aligned16(a_bf16) || !aligned16(b_packed) || !aligned16(c_bf16))
    return MXFP4_ERR_INVALID_ARG;
  mxfp4::GemmPlan plan;
  if (mxfp4::make_gemm_plan(m, n, k, &plan) != 0) return MXFP4_ERR_UNSUPPORTED;
  if (plan.workspace > 0) {
    if (!workspace || workspace_bytes < plan.workspace) return MXFP4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MXFP4_ERR_INVALID_ARG;
  }
  return from_cuda(mxfp4::launch_gemm(plan, a_bf16, m, k, lda, b_packed, n, c_bf16, ldc, workspace,
                                      static_cast<cudaStream_t>(stream)));
}

mxfp4_status mxfp4_gemm_host(const void* a_host, int64_t m, int64_t k, int64_t lda, const void* b_packed, int64_t n,
                             void* c_host, int64_t ldc, void* a_dev, void* c_dev, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (m <= 0 || n <= 0 || !valid_k(k) || lda < k || ldc < n) return MXFP4_ERR_INVALID_ARG;
  if (!a_host || !c_host || !a_dev || !c_dev || !aligned16(a_dev) || !aligned16(c_dev)) return MXFP4_ERR_INVALID_ARG;
  const int64_t n8 = (n + 7) & ~int64_t(7);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t esz = 2;  // bf16
  // validate everything the GEMM checks before enqueueing the first copy
  mxfp4::GemmPlan plan;
  if (!b_packed || !aligned16(b_packed)) return MXFP4_ERR_INVALID_ARG;
  if (mxfp4::make_gemm_plan(m, n, k, &plan) != 0) return MXFP4_ERR_UNSUPPORTED;
  if (plan.workspace > 0 && (!workspace || workspace_bytes < plan.workspace)) return MXFP4_ERR_WORKSPACE;
  if (plan.workspace > 0 && !aligned16(workspace)) return MXFP4_ERR_INVALID_ARG;
  // The fused small-m kernel, the activation quantizer and the one-CTA
  // GEMMs read A with plain loads and write C with plain stores, so with
  // page-locked buffers they work on host memory directly (NVLink-C2C on
  // GB300): no copy on either side.  Not the CTA-pair plan, whose C goes out
  // through tensor-map bulk stores, and not the fused kernel beyond one
  // round of A loads per CTA: each further round waits a host-memory round
  // trip (m = 16, k = 7168 measured 48 us this way against 27 us with the
  // two copies; m = 32, k = 512 10-20 us, as fast as or faster than the
  // copies; m = 64, k = 2048 17 us against 36 us; m = 256, k = 1536 23 us
  // against 38 us).
  const bool direct = plan.mode == 0 ? k <= kDirectHostMaxK : !plan.persistent;
  if (direct) {
    const void* a_map = mapped_host(a_host);
    void* c_map = a_map ? mapped_host(c_host) : nullptr;
    if (a_map && c_map && aligned16(a_map) && aligned16(c_map) && (lda % 8) == 0 && (ldc % 8) == 0)
      return mxfp4_gemm(a_map, m, k, lda, b_packed, n, c_map, ldc, workspace, workspace_bytes, stream);
  }
  const auto* ah = static_cast<const uint8_t*>(a_host);
  auto* ch = static_cast<uint8_t*>(c_host);
  auto* ad = static_cast<uint8_t*>(a_dev);
  auto* cd = static_cast<uint8_t*>(c_dev);
  HostPipe* hp = nullptr;
  if (m > 32 && static_cast<size_t>(m) * static_cast<size_t>(n) * esz >= kChunkMinCBytes && m >= 2 * kChunkRowAlign) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MXFP4_ERR_CUDA;
    hp = host_pipe(cap == cudaStreamCaptureStatusNone);
  }
  if (!hp) {
    if (cudaMemcpy2DAsync(a_dev, k * esz, a_host, lda * esz, k * esz, m, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MXFP4_ERR_CUDA;
    const mxfp4_status s = mxfp4_gemm(a_dev, m, k, k, b_packed, n, c_dev, n8, workspace, workspace_bytes, stream);
    if (s != MXFP4_OK) return s;
    return from_cuda(cudaMemcpy2DAsync(c_host, ldc * esz, c_dev, n8 * esz, n * esz, m, cudaMemcpyDeviceToHost, st));
  }
  // chunked: up, GEMM, (fork) down, per chunk of rows; the caller's stream
  // waits for the last download before anything enqueued after this call
  int64_t rows = (m + kMaxChunks - 1) / kMaxChunks;
  rows = (rows + kChunkRowAlign - 1) / kChunkRowAlign * kChunkRowAlign;
  int i = 0;
  for (int64_t r0 = 0; r0 < m; r0 += rows, ++i) {
    const int64_t mr = m - r0 < rows ? m - r0 : rows;
    if (cudaMemcpy2DAsync(ad + r0 * k * esz, k * esz, ah + r0 * lda * esz, lda * esz, k * esz, mr,
                          cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MXFP4_ERR_CUDA;
    const mxfp4_status s = mxfp4_gemm(ad + r0 * k * esz, mr, k, k, b_packed, n, cd + r0 * n8 * esz, n8, workspace,
                                      workspace_bytes, stream);
    if (s != MXFP4_OK) return s;
    if (cudaEventRecord(hp->ev[i], st) != cudaSuccess || cudaStreamWaitEvent(hp->stream, hp->ev[i], 0) != cudaSuccess ||
        cudaMemcpy2DAsync(ch + r0 * ldc * esz, ldc * esz, cd + r0 * n8 * esz, n8 * esz, n * esz, mr,
                          cudaMemcpyDeviceToHost, hp->stream) != cudaSuccess)
      return MXFP4_ERR_CUDA;
  }
  if (cudaEventRecord(hp->ev[kMaxChunks], hp->stream) != cudaSuccess) return MXFP4_ERR_CUDA;
  return from_cuda(cudaStreamWaitEvent(st, hp->ev[kMaxChunks], 0));
}

mxfp4_status mxfp4_prepack_b_bf16(const void* b_bf16, int64_t n, int64_t k, int64_t ldb, void* b_packed,
                                  size_t b_packed_bytes, void* stream) {
  if (n <= 0 || !valid_k(k) || ldb < k || (ldb % 8) != 0) return MXFP4_ERR_INVALID_ARG;
  if (!b_bf16 || !b_packed || !aligned16(b_bf16) || !aligned16(b_packed)) return MXFP4_ERR_INVALID_ARG;
  if (b_packed_bytes < mxfp4_prepacked_b_bytes(n, k)) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(mxfp4::launch_quant_image(b_bf16, n, k, ldb, b_packed, static_cast<cudaStream_t>(stream),
                                             /*zero_padding_rows=*/true));
}

size_t mxfp4_act_image_bytes(int64_t m, int64_t k) {
  if (m <= 0 || !valid_k(k)) return 0;
  return static_cast<size_t>(mxfp4::image_bytes(m, k));
}

mxfp4_status mxfp4_quant_image(const void* a_bf16, int64_t m, int64_t k, int64_t lda, void* a_image,
                               size_t a_image_bytes, void* stream) {
  if (m <= 0 || !valid_k(k) || lda < k || (lda % 8) != 0) return MXFP4_ERR_INVALID_ARG;
  if (!a_bf16 || !a_image || !aligned16(a_bf16) || !aligned16(a_image)) return MXFP4_ERR_INVALID_ARG;
  if (a_image_bytes < mxfp4_act_image_bytes(m, k)) return MXFP4_ERR_INVALID_ARG;
  return from_cuda(mxfp4::launch_quant_image(a_bf16, m, k, lda, a_image, static_cast<cudaStream_t>(stream)));
}

mxfp4_status mxfp4_gemm_image(const void* a_image, int64_t m, int64_t k, const void* b_packed, int64_t n,
                              void* c_bf16, int64_t ldc, void* stream) {
  if (m <= 0 || n <= 0 || !valid_k(k) || ldc < n || (ldc % 8) != 0) return MXFP4_ERR_INVALID_ARG;
  if (!a_image || !b_packed || !c_bf16 || !aligned16(a_image) || !aligned16(b_packed) || !aligned16(c_bf16))
    return MXFP4_ERR_INVALID_ARG;
  mxfp4::GemmPlan plan;
  if (mxfp4::make_gemm_plan(m, n, k, &plan, /*a_image=*/true) != 0) return MXFP4_ERR_UNSUPPORTED;
  return from_cuda(mxfp4::launch_gemm(plan, nullptr, m, k, k, b_packed, n, c_bf16, ldc, nullptr,
                                      static_cast<cudaStream_t>(stream), a_image));
}

mxfp4_status mxfp4_set_debug_options(int split_k, int drop_copies) {
  return mxfp4::set_debug_options(split_k, drop_copies) ? MXFP4_OK : MXFP4_ERR_INVALID_ARG;
}

mxfp4_status mxfp4_kernel_binary_version(int* version) {
  if (!version) return MXFP4_ERR_INVALID_ARG;
  const int v = mxfp4::kernel_binary_version();
  if (v < 0) {
    (void)cudaGetLastError();
    return MXFP4_ERR_CUDA;
  }
  *version = v;
  return MXFP4_OK;
}

mxfp4_status mxfp4_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MXFP4_ERR_CUDA;
  int flag = 0;
  if (mxfp4::read_and_clear_timeout_flag(&flag) != cudaSuccess) return MXFP4_ERR_CUDA;
  return flag ? MXFP4_ERR_TIMEOUT : MXFP4_OK;
}

}  // extern "C"
