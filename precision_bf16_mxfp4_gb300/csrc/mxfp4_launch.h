// Internal host-side declarations shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mxfp4 {

// The e2m1 conversion used by every quantizing kernel: false selects the
// midpoint-comparison encoder, true the cvt.rn.satfinite.e2m1x2 instruction
// (round to nearest even, saturating at 6; its first source operand lands in
// the upper nibble).  Both agree with the oracle bit for bit on every finite
// bf16 value times every block exponent with |q| < 8; the GPU tests check the
// selected one on every run.
constexpr bool kUseHardwareCvt = true;

int num_sms();  // multiprocessors of the current device (cached per device)

cudaError_t launch_quant_linear(const void* a, int64_t m, int64_t k, int64_t lda, void* q, void* scale,
                                cudaStream_t stream);
cudaError_t launch_quant_image(const void* a, int64_t m, int64_t k, int64_t lda, void* img, cudaStream_t stream,
                               bool zero_padding_rows = false);
cudaError_t launch_prepack(const void* bq, const void* bs, int64_t n, int64_t k, void* img, cudaStream_t stream);

// GEMM execution plan chosen from (m, n, k) and the device.
struct GemmPlan {
  int mode;            // 0: swap-AB, A quantized in the GEMM; 1: swap-AB on A's image; 2: A image x weights
  bool swap_ab;        // weights on the MMA's 128-row side
  int bn;              // MMA N: padded m (swap) or the n tile (no swap)
  int split;           // CTAs per cluster splitting K
  bool persistent;     // CTA pairs (one per two SMs) looping over 256 x 256 tiles (plain mode, many tiles)
  int64_t grid_x;      // 128-row tiles of the MMA-A operand
  int64_t grid_y;      // N tiles times split
  size_t workspace;    // bytes of caller workspace the plan needs
};

// a_image: the activation arrives as an operand image already (image modes
// only, no workspace).  Returns 0 = ok, else unsupported.
int make_gemm_plan(int64_t m, int64_t n, int64_t k, GemmPlan* plan, bool a_image = false);
// With a_image non-null the GEMM reads that activation image instead of
// quantizing a_bf16 into the workspace.
cudaError_t launch_gemm(const GemmPlan& plan, const void* a_bf16, int64_t m, int64_t k, int64_t lda,
                        const void* b_image, int64_t n, void* c, int64_t ldc, void* workspace,
                        cudaStream_t stream, const void* a_image = nullptr);

// Device-side watchdog flag: set by a kernel whose bounded wait ran out.
cudaError_t read_and_clear_timeout_flag(int* flag);

// Testing and tuning overrides (K split 0/1/2/4/8, copy dropping 0/1);
// false for values outside those sets.
bool set_debug_options(int split_k, int drop_copies);

// binaryVersion of the small-m GEMM kernel as loaded on the current device
// (major * 10 + minor), or -1 if the query failed.
int kernel_binary_version();

}  // namespace mxfp4
