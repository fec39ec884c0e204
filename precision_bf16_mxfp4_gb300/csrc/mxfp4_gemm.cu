// MXFP4 GEMM  C[m,n] = quant(A) . B^T  on tcgen05 block-scaled tensor cores.
//
// Semantics (kernelbot amd-mxfp4-mm pages, submission 752099: the
// `tl.dot_scaled(a, a_scale, "e2m1", b, b_scale, "e2m1", acc)` product with
// fp32 accumulation and a bf16 result; submission 694791 for the quantizer):
//   C[i,j] = bf16( sum_kb 2^(sa[i,kb]-127) 2^(sb[j,kb]-127) sum_t a[i,32kb+t] b[j,32kb+t] )
//
// One CTA computes a 128 x BN accumulator tile in tensor memory.  The MMA's
// 128-row operand ("MMA-A") always comes from a tiled operand image through
// bulk copies.  Two modes:
//   swap-AB, fused (m <= 64): MMA-A = the prepacked weight image (n on the
//     128-row side); MMA-B = the activations, quantized by producer warps
//     straight from bf16 into shared memory in the MMA layout (quantized A
//     never reaches HBM); BN = m padded to 16/32/64.
//   plain (m > 64): MMA-A = the activation image written by
//     quant_image_kernel into the workspace; MMA-B = BN/128 weight tiles.
// K may be split across the CTAs of a thread-block cluster; their fp32
// partial tiles are summed in a fixed order through distributed shared memory.
//
// Warp roles: warp 0 issues bulk copies; warp 1 owns tensor memory and issues
// scale-factor copies and MMAs (one thread); warps 2-5 run the epilogue; in
// the fused mode warps 2-7 also quantize the activations.  Every wait is
// bounded: a wait that runs out sets a device flag and the CTA winds down.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_launch.h"
#include "ptx.cuh"

namespace mxfp4 {

__device__ int g_timeout_flag = 0;

constexpr uint64_t kWaitLimitNs = 1000000000ull;    // 1 s for a pipeline wait
constexpr uint64_t kDrainLimitNs = 20000000ull;     // 20 ms when winding down after a timeout
constexpr int kStages = 4;
constexpr int kQuantWarps = 6;

struct GemmArgs {
  const uint8_t* a_img;  // MMA-A operand image
  int64_t a_rows;        // rows of the matrix in a_img
  const uint8_t* b_img;  // MMA-B weight image (plain mode)
  int64_t b_rows;        // rows of the matrix in b_img
  const uint16_t* act;   // bf16 activations (fused mode)
  int64_t lda;
  int64_t m, n, k;
  int64_t kt_count;      // K tiles of 256
  __nv_bfloat16* c;
  int64_t ldc;
  int split;
};

template <int BN, bool kFused>
struct Cfg {
  static constexpr int kThreads = kFused ? 32 * (2 + kQuantWarps) : 32 * 6;
  static constexpr int kBTiles = kFused ? 1 : BN / 128;           // weight tiles per stage (plain)
  static constexpr int kBDataBytes = BN * 128;
  static constexpr int kBSfBytes = kBTiles * kTileSfBytes;
  static constexpr int kOffAData = 0;
  static constexpr int kOffBData = kOffAData + kStages * kTileDataBytes;
  static constexpr int kOffASf = kOffBData + kStages * kBDataBytes;
  static constexpr int kOffBSf = kOffASf + kStages * kTileSfBytes;
  static constexpr int kOffBars = kOffBSf + kStages * kBSfBytes;
  static constexpr int kOffMisc = kOffBars + (2 * kStages + 1) * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr int kRedStride = BN + 4;                 // fp32 partial tile row stride
  static_assert(128 * kRedStride * 4 <= kOffBars, "split-K partial tile must fit in the stage buffers");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // tensor memory: accumulator columns, then per-stage scale-factor columns
  static constexpr int kAccCols = BN;
  static constexpr int kSfbColsPerGroup = 4 * ((BN + 127) / 128);
  static constexpr int kSfColsPerStage = 8 + 2 * kSfbColsPerGroup;
  static constexpr int kTmemNeed = kAccCols + kStages * kSfColsPerStage;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "tensor memory");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
};

__device__ __forceinline__ void raise_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(&g_timeout_flag, 1);
}

// Wait for phase `parity` of `bar`; false if the CTA is aborting or the
// wait ran past its limit (which starts the abort).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        raise_timeout(abort_flag);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int BN, bool kFused>
__global__ void __launch_bounds__(Cfg<BN, kFused>::kThreads, 1) gemm_kernel(const GemmArgs args) {
  using C = Cfg<BN, kFused>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = args.split;
  const int rank = split > 1 ? (int)(blockIdx.y % split) : 0;
  const int64_t a_tile = blockIdx.x;
  const int64_t b_tile = blockIdx.y / split;
  const int64_t KT = args.kt_count;
  const int64_t kt_begin = KT * rank / split;
  const int64_t kt_end = KT * (rank + 1) / split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1 + (kFused ? kQuantWarps * 32 : 0));
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ bulk-copy producer
    if (lane == 0) {
      const uint64_t policy_stream = policy_evict_first();
      const uint8_t* a_sf_region = args.a_img + image_sf_region(args.a_rows, args.k);
      const int64_t b_row_tiles = kFused ? 0 : ceil_div(args.b_rows, kTileRows);
      const uint8_t* b_sf_region = kFused ? nullptr : args.b_img + image_sf_region(args.b_rows, args.k);
      uint32_t issued_parity[kStages];
      bool used[kStages];
      for (int s = 0; s < kStages; ++s) used[s] = false;
      if (!kFused) pdl_wait();  // the activation image comes from the preceding kernel
      int s = 0;
      uint32_t ph = 0;
      for (int64_t kt = kt_begin; kt < kt_end; ++kt) {
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag)) break;
        uint32_t bytes = kTileDataBytes + kTileSfBytes;
        if (!kFused) {
          for (int t = 0; t < C::kBTiles; ++t)
            if (b_tile * C::kBTiles + t < b_row_tiles) bytes += kTileDataBytes + kTileSfBytes;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        const int64_t at = a_tile * KT + kt;
        if (kFused) {
          bulk_load_hint(smem + C::kOffAData + s * kTileDataBytes, args.a_img + at * kTileDataBytes,
                         kTileDataBytes, &full[s], policy_stream);
          bulk_load_hint(smem + C::kOffASf + s * kTileSfBytes, a_sf_region + at * kTileSfBytes, kTileSfBytes,
                         &full[s], policy_stream);
        } else {
          bulk_load(smem + C::kOffAData + s * kTileDataBytes, args.a_img + at * kTileDataBytes, kTileDataBytes,
                    &full[s]);
          bulk_load(smem + C::kOffASf + s * kTileSfBytes, a_sf_region + at * kTileSfBytes, kTileSfBytes,
                    &full[s]);
          for (int t = 0; t < C::kBTiles; ++t) {
            const int64_t brt = b_tile * C::kBTiles + t;
            if (brt >= b_row_tiles) continue;
            const int64_t bt = brt * KT + kt;
            bulk_load(smem + C::kOffBData + s * C::kBDataBytes + t * kTileDataBytes,
                      args.b_img + bt * kTileDataBytes, kTileDataBytes, &full[s]);
            bulk_load(smem + C::kOffBSf + s * C::kBSfBytes + t * kTileSfBytes, b_sf_region + bt * kTileSfBytes,
                      kTileSfBytes, &full[s]);
          }
        }
        issued_parity[s] = ph;
        used[s] = true;
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (*abort_flag) {  // let copies already in flight land before the CTA exits
        for (int t = 0; t < kStages; ++t)
          if (used[t]) wait_bounded(&full[t], issued_parity[t], abort_flag, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool accumulate = false;
      for (int64_t kt = kt_begin; kt < kt_end; ++kt) {
        if (!wait_bounded(&full[s], ph, abort_flag)) break;
        tc_fence_after();
        const uint32_t sfa = tmem + C::kAccCols + s * C::kSfColsPerStage;
        const uint32_t sfb = sfa + 8;
        const uint32_t a_sf_s = smem_addr(smem + C::kOffASf + s * kTileSfBytes);
        const uint32_t b_sf_s = smem_addr(smem + C::kOffBSf + s * C::kBSfBytes);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          tmem_copy_32x128b_x4(sfa + g * 4, smem_desc(a_sf_s + g * kAtomBytes, 0, 128, kLayoutNoSwizzle));
#pragma unroll
          for (int h = 0; h < C::kSfbColsPerGroup / 4; ++h)
            tmem_copy_32x128b_x4(sfb + g * C::kSfbColsPerGroup + h * 4,
                                 smem_desc(b_sf_s + h * kTileSfBytes + g * kAtomBytes, 0, 128, kLayoutNoSwizzle));
        }
        const uint32_t a_s = smem_addr(smem + C::kOffAData + s * kTileDataBytes);
        const uint32_t b_s = smem_addr(smem + C::kOffBData + s * C::kBDataBytes);
        const int64_t rem = args.k - kt * kTileK;
        const int kk_count = rem >= kTileK ? 4 : (int)ceil_div(rem, 64);
        for (int kk = 0; kk < kk_count; ++kk) {
          const int g = kk >> 1;
          const uint32_t id = (uint32_t)(kk & 1) * 2;
          mma_mxf4(tmem, smem_desc(a_s + kk * 32, 0, 1024, kLayoutSwizzle128),
                   smem_desc(b_s + kk * 32, 0, 1024, kLayoutSwizzle128), idesc_mxf4(128, BN, id, id),
                   sfa + g * 4, sfb + g * C::kSfbColsPerGroup, accumulate ? 1u : 0u);
          accumulate = true;
        }
        mma_commit(&empty[s]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      mma_commit(accum);  // fires once every MMA above has completed
    }
    __syncwarp();
  }

  if constexpr (kFused) {
    // ---------------------------------------- activation quantizers (warps 2-7)
    if (warp >= 2) {
      constexpr int kRowsPerWarp = (BN + kQuantWarps - 1) / kQuantWarps;
      const int qw = warp - 2;
      int s = 0;
      uint32_t ph = 0;
      for (int64_t kt = kt_begin; kt < kt_end; ++kt) {
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag)) break;
        uint8_t* bd = smem + C::kOffBData + s * C::kBDataBytes;
        uint8_t* bsf = smem + C::kOffBSf + s * C::kBSfBytes;
        const int64_t col = kt * kTileK + lane * 8;
        uint4 w[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const int row = qw + i * kQuantWarps;
          w[i] = (row < args.m && col < args.k) ? ldg_nc_v4(args.act + row * args.lda + col)
                                                : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const int row = qw + i * kQuantWarps;
          if (row < BN) {  // uniform across the warp
            uint32_t sbyte;
            const uint32_t packed = quantize_lane<kUseHardwareCvt>(w[i], sbyte);
            *reinterpret_cast<uint32_t*>(bd + tile_data_offset(row, lane * 4)) = packed;
            if ((lane & 3) == 0) bsf[tile_sf_offset(row, lane >> 2)] = (uint8_t)sbyte;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&full[s]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  }

  // ------------------------------------------------------------- epilogue
  float* red = reinterpret_cast<float*>(smem);  // split-K partial tile (stage buffers are idle now)
  if (warp >= 2 && warp < 6) {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // accumulator row = tensor-memory lane
    const bool ok = wait_bounded(accum, 0, abort_flag);
    tc_fence_after();
    if (ok) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t r[16];
        tmem_load_16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, r);
        tmem_load_wait();
        if (split > 1) {
          float4* dst = reinterpret_cast<float4*>(red + row * C::kRedStride + c0);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        } else if (kFused) {
          const int64_t n_idx = a_tile * kTileRows + row;
          if (n_idx < args.n) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int64_t m_idx = c0 + j;
              if (m_idx < args.m) args.c[m_idx * args.ldc + n_idx] = __float2bfloat16_rn(__uint_as_float(r[j]));
            }
          }
        } else {
          const int64_t m_idx = a_tile * kTileRows + row;
          const int64_t n0 = b_tile * BN + c0;
          if (m_idx < args.m) {
            __nv_bfloat16* dst = args.c + m_idx * args.ldc + n0;
            if (n0 + 16 <= args.n) {
              uint4 v0, v1;
              v0.x = bf16x2_bits(__uint_as_float(r[0]), __uint_as_float(r[1]));
              v0.y = bf16x2_bits(__uint_as_float(r[2]), __uint_as_float(r[3]));
              v0.z = bf16x2_bits(__uint_as_float(r[4]), __uint_as_float(r[5]));
              v0.w = bf16x2_bits(__uint_as_float(r[6]), __uint_as_float(r[7]));
              v1.x = bf16x2_bits(__uint_as_float(r[8]), __uint_as_float(r[9]));
              v1.y = bf16x2_bits(__uint_as_float(r[10]), __uint_as_float(r[11]));
              v1.z = bf16x2_bits(__uint_as_float(r[12]), __uint_as_float(r[13]));
              v1.w = bf16x2_bits(__uint_as_float(r[14]), __uint_as_float(r[15]));
              reinterpret_cast<uint4*>(dst)[0] = v0;
              reinterpret_cast<uint4*>(dst)[1] = v1;
            } else {
              for (int j = 0; j < 16 && n0 + j < args.n; ++j) dst[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();

  if (split > 1) {
    // -------------------------- split-K: fixed-order sum over the cluster's partials
    cluster_sync();
    const int rows = kTileRows / split;
    const int row0 = rank * rows;
    constexpr int kC4 = BN / 4;
    const uint32_t red_addr = smem_addr(red);
    for (int g = threadIdx.x; g < rows * kC4; g += C::kThreads) {
      const int rr = g % rows, c4 = g / rows;
      const int row = row0 + rr;
      const uint32_t off = (uint32_t)((row * C::kRedStride + c4 * 4) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < split; ++q) {
        const float4 v = ld_cluster_f4(map_cluster(red_addr, (uint32_t)q) + off);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
      if (kFused) {
        const int64_t n_idx = a_tile * kTileRows + row;
        if (n_idx < args.n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t m_idx = c4 * 4 + e;
            if (m_idx < args.m) args.c[m_idx * args.ldc + n_idx] = __float2bfloat16_rn(vals[e]);
          }
        }
      } else {
        const int64_t m_idx = a_tile * kTileRows + row;
        const int64_t n0 = b_tile * BN + c4 * 4;
        if (m_idx < args.m) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n0 + e < args.n) args.c[m_idx * args.ldc + n0 + e] = __float2bfloat16_rn(vals[e]);
        }
      }
    }
    cluster_sync();  // keep every partial tile alive until all ranks have read it
  }

  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host
int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 148;
  }
  return cached[dev];
}

int make_gemm_plan(int64_t m, int64_t n, int64_t k, GemmPlan* plan) {
  const int sms = num_sms();
  const int64_t KT = ceil_div(k, kTileK);
  GemmPlan p{};
  if (m <= 64) {
    p.swap_ab = true;
    p.bn = m <= 16 ? 16 : (m <= 32 ? 32 : 64);
    p.grid_x = ceil_div(n, kTileRows);
    int s = 1;
    while (s < 8 && p.grid_x * s * 2 <= sms && KT / (s * 2) >= 1) s *= 2;
    p.split = s;
    p.grid_y = s;
    p.workspace = 0;
  } else {
    p.swap_ab = false;
    const int64_t mt = ceil_div(m, kTileRows);
    p.bn = (mt * ceil_div(n, 256) >= sms) ? 256 : 128;
    p.grid_x = mt;
    const int64_t nt = ceil_div(n, p.bn);
    int s = 1;
    while (s < 8 && mt * nt * s * 2 <= sms && KT / (s * 2) >= 2) s *= 2;
    p.split = s;
    p.grid_y = nt * s;
    p.workspace = (size_t)image_bytes(m, k);
  }
  if (p.grid_x > 0x7FFFFFFF || p.grid_y > 65535) return 1;
  *plan = p;
  return 0;
}

template <int BN, bool kFused>
static cudaError_t launch_one(const GemmPlan& plan, const GemmArgs& args, cudaStream_t stream, bool pdl) {
  using C = Cfg<BN, kFused>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)plan.grid_x, (unsigned)plan.grid_y, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (plan.split > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = (unsigned)plan.split;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN, kFused>, args);
}

cudaError_t launch_gemm(const GemmPlan& plan, const void* a_bf16, int64_t m, int64_t k, int64_t lda,
                        const void* b_image, int64_t n, void* c, int64_t ldc, void* workspace,
                        cudaStream_t stream) {
  GemmArgs args{};
  args.m = m;
  args.n = n;
  args.k = k;
  args.kt_count = ceil_div(k, kTileK);
  args.c = static_cast<__nv_bfloat16*>(c);
  args.ldc = ldc;
  args.split = plan.split;
  args.lda = lda;
  if (plan.swap_ab) {
    args.a_img = static_cast<const uint8_t*>(b_image);
    args.a_rows = n;
    args.act = static_cast<const uint16_t*>(a_bf16);
    switch (plan.bn) {
      case 16: return launch_one<16, true>(plan, args, stream, false);
      case 32: return launch_one<32, true>(plan, args, stream, false);
      case 64: return launch_one<64, true>(plan, args, stream, false);
      default: return cudaErrorInvalidValue;
    }
  }
  cudaError_t e = launch_quant_image(a_bf16, m, k, lda, workspace, stream);
  if (e != cudaSuccess) return e;
  args.a_img = static_cast<const uint8_t*>(workspace);
  args.a_rows = m;
  args.b_img = static_cast<const uint8_t*>(b_image);
  args.b_rows = n;
  switch (plan.bn) {
    case 128: return launch_one<128, false>(plan, args, stream, true);
    case 256: return launch_one<256, false>(plan, args, stream, true);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t read_and_clear_timeout_flag(int* flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_timeout_flag, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_timeout_flag, &zero, sizeof(int));
}

}  // namespace mxfp4
