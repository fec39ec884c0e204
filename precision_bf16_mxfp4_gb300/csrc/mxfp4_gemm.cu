// MXFP4 GEMM  C[m,n] = quant(A) . B^T  on tcgen05 block-scaled tensor cores.
//
// Semantics (kernelbot amd-mxfp4-mm pages, submission 752099: the
// `tl.dot_scaled(a, a_scale, "e2m1", b, b_scale, "e2m1", acc)` product with
// fp32 accumulation and a bf16 result; submission 694791 for the quantizer):
//   C[i,j] = bf16( sum_kb 2^(sa[i,kb]-127) 2^(sb[j,kb]-127) sum_t a[i,32kb+t] b[j,32kb+t] )
//
// One CTA computes a 128 x BN accumulator tile in tensor memory.  The MMA's
// 128-row operand ("MMA-A") comes from a tiled operand image through bulk
// copies.  Three modes:
//   kFusedSwap (m <= 32): swap-AB.  MMA-A = prepacked weights (n on the
//     128-row side); MMA-B = the activations, quantized by producer warps
//     from bf16 straight into shared memory in the MMA operand and scale
//     layouts, so quantized A never reaches HBM.  BN = m padded to 16/32.
//   kImageSwap (32 < m <= 128): swap-AB; MMA-B = the first BN rows of the
//     activation image that quant_image_kernel wrote into the workspace.
//   kImagePlain (m > 128): MMA-A = activation image, MMA-B = BN/128 weight
//     tiles.
// In the image modes the GEMM is launched as a programmatic dependent of the
// quantization kernel: it prefetches the weight stages first and waits for
// the activation image only before loading it.
//
// K may be split across the S CTAs of a thread-block cluster.  Rank r owns
// accumulator rows [128r/S, 128(r+1)/S): every rank writes those rows of its
// fp32 partial into slot r of the owner's shared memory (st.shared::cluster;
// its own rows locally) and the other ranks arrive on the owner's mbarrier
// with cluster-scope release, one arrival per warp; the owner adds the S
// slots in rank order (deterministic) and stores its rows.
//
// Warp roles: warp 0 issues bulk copies; warp 1 owns tensor memory and issues
// scale-factor copies and MMAs (one thread); warps 2-5 drain the accumulator;
// in kFusedSwap warps 2-7 quantize the activations.  All threads stage and
// store the bf16 output with 16-byte coalesced writes.  Every wait is
// bounded: a wait that runs out sets a device flag and the CTA winds down.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "mxfp4_device.cuh"
#include "mxfp4_launch.h"
#include "ptx.cuh"

namespace mxfp4 {

__device__ int g_timeout_flag = 0;

// Wait limits in SM clock cycles (read with clock64, which costs a few
// cycles, unlike the global timer): 2^31 cycles is about 1 s at 2 GHz.
constexpr long long kWaitLimitCycles = 1ll << 31;
constexpr long long kDrainLimitCycles = 1ll << 25;  // ~20 ms when winding down after a timeout
constexpr int kStages = 4;
constexpr int kQuantWarps = 6;

enum GemmMode : int { kFusedSwap = 0, kImageSwap = 1, kImagePlain = 2 };

struct GemmArgs {
  const uint8_t* a_img;  // MMA-A operand image
  int64_t a_rows;        // rows of the matrix in a_img
  const uint8_t* b_img;  // MMA-B operand image (image modes)
  int64_t b_rows;        // rows of the matrix in b_img
  const uint16_t* act;   // bf16 activations (kFusedSwap)
  int64_t lda;
  int64_t m, n, k;
  int64_t kt_count;  // K tiles of 256
  __nv_bfloat16* c;
  int64_t ldc;
  int split;
};

template <int BN, int kMode>
struct Cfg {
  static constexpr bool kFused = kMode == kFusedSwap;
  static constexpr bool kSwap = kMode != kImagePlain;
  static constexpr int kThreads = kFused ? 32 * (2 + kQuantWarps) : 32 * 6;
  static constexpr int kBTiles = (BN + 127) / 128;          // image tiles feeding MMA-B per stage
  static constexpr int kBRowsPerTile = BN < 128 ? BN : 128;  // rows taken from each of them
  static constexpr int kBDataBytes = BN * 128;
  static constexpr int kBSfBytes = kBTiles * kTileSfBytes;
  static constexpr int kOffAData = 0;
  static constexpr int kOffBData = kOffAData + kStages * kTileDataBytes;
  static constexpr int kOffASf = kOffBData + kStages * kBDataBytes;
  static constexpr int kOffBSf = kOffASf + kStages * kTileSfBytes;
  static constexpr int kOffBars = kOffBSf + kStages * kBSfBytes;
  static constexpr int kOffMisc = kOffBars + (2 * kStages + 2) * 8;
  // K split across a cluster: rank r owns accumulator rows [r*128/S, (r+1)*128/S);
  // every other rank pushes those rows of its fp32 partial into the owner's
  // shared memory, in a region of its own (a rank may push while the owner's
  // MMAs still read the stage buffers).
  static constexpr int kMaxSplit = (kMode == kImagePlain && BN == 256) ? 1 : 8;
  static constexpr int kRedStride = BN + 4;  // fp32 partial-row pitch (floats)
  static constexpr int kRedBytes = kMaxSplit > 1 ? 128 * kRedStride * 4 : 0;  // [S][128/S][kRedStride]
  static constexpr int kOffRed = (kOffMisc + 16 + 15) & ~15;
  static constexpr int kSmemBytes = kOffRed + kRedBytes + 1024;  // + alignment slack
  // bf16 output staging reuses the stage buffers once the accumulator is complete
  static constexpr int kStgPitch = kSwap ? 128 : BN + 8;  // elements
  static constexpr int kStgBytes = (kSwap ? BN : 128) * kStgPitch * 2;
  static_assert(kStgBytes <= kOffBars, "output staging must fit in the stage buffers");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // tensor memory: accumulator columns, then per-stage scale-factor columns
  static constexpr int kAccCols = BN;
  static constexpr int kSfbColsPerGroup = 4 * kBTiles;
  static constexpr int kSfColsPerStage = 8 + 2 * kSfbColsPerGroup;
  static constexpr int kTmemNeed = kAccCols + kStages * kSfColsPerStage;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "tensor memory");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(!kSwap || BN <= 128, "swap-AB keeps the activations in one image tile");
  static_assert(!kFused || BN <= 8 * kQuantWarps * 8, "quantizer rows");
};

__device__ __forceinline__ void raise_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(&g_timeout_flag, 1);
}

// Wait for phase `parity` of `bar`; false if the CTA is aborting or the
// wait ran past its limit (which starts the abort).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             long long limit_cycles = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit_cycles) {
        raise_timeout(abort_flag);
        return false;
      }
    }
  }
}

// Same, acquiring at cluster scope (for phases completed by other CTAs' arrivals).
__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
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

template <int BN, int kMode>
__global__ void __launch_bounds__(Cfg<BN, kMode>::kThreads, 1) gemm_kernel(const GemmArgs args) {
  using C = Cfg<BN, kMode>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint64_t* red_full = accum + 1;  // rank 0: all other ranks' partial rows have landed
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
  const int nk = (int)(kt_end - kt_begin);

  // ------------------------------------------------ copy issue (warp 0, lane 0)
  const uint8_t* a_sf_region = args.a_img + image_sf_region(args.a_rows, args.k);
  const int64_t b_row_tiles = C::kFused ? 0 : ceil_div(args.b_rows, kTileRows);
  const uint8_t* b_sf_region = C::kFused ? nullptr : args.b_img + image_sf_region(args.b_rows, args.k);
  auto stage_bytes = [&]() -> uint32_t {
    uint32_t bytes = kTileDataBytes + kTileSfBytes;
    if (!C::kFused)
      for (int t = 0; t < C::kBTiles; ++t)
        if (b_tile * C::kBTiles + t < b_row_tiles) bytes += C::kBRowsPerTile * 128 + kTileSfBytes;
    return bytes;
  };
  auto issue_a = [&](int64_t kt, int s, uint64_t policy) {
    const int64_t at = a_tile * KT + kt;
    bulk_load_hint(smem + C::kOffAData + s * kTileDataBytes, args.a_img + at * kTileDataBytes, kTileDataBytes,
                   &full[s], policy);
    bulk_load_hint(smem + C::kOffASf + s * kTileSfBytes, a_sf_region + at * kTileSfBytes, kTileSfBytes, &full[s],
                   policy);
  };
  auto issue_b = [&](int64_t kt, int s, uint64_t policy) {
    for (int t = 0; t < C::kBTiles; ++t) {
      const int64_t brt = b_tile * C::kBTiles + t;
      if (brt >= b_row_tiles) continue;
      const int64_t bt = brt * KT + kt;
      bulk_load_hint(smem + C::kOffBData + s * C::kBDataBytes + t * kTileDataBytes,
                     args.b_img + bt * kTileDataBytes, C::kBRowsPerTile * 128, &full[s], policy);
      bulk_load_hint(smem + C::kOffBSf + s * C::kBSfBytes + t * kTileSfBytes, b_sf_region + bt * kTileSfBytes,
                     kTileSfBytes, &full[s], policy);
    }
  };
  // which operand the preceding quantization kernel produces
  constexpr bool kADependent = kMode == kImagePlain;
  constexpr bool kBDependent = kMode == kImageSwap;

  uint64_t pol_weights = 0, pol_act = 0;
  if (threadIdx.x == 0) {
    // The weight stream is the long pole: initialize only the stage-full
    // barriers, start the first stages' copies, then set up the rest.
    // Operands written by the preceding kernel are requested only after the
    // programmatic-dependency wait.
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1 + (C::kFused ? kQuantWarps * 32 : 0));
    fence_mbar_init();
    pol_weights = policy_evict_first();
    pol_act = policy_evict_last();
    const int pre = nk < kStages ? nk : kStages;
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], stage_bytes());
      if (!kADependent) issue_a(kt_begin + i, i, kMode == kImagePlain ? pol_act : pol_weights);
      if (!C::kFused && !kBDependent) issue_b(kt_begin + i, i, pol_weights);
    }
    for (int s = 0; s < kStages; ++s) mbar_init(&empty[s], 1);
    mbar_init(accum, 1);
    // one arrival per (other rank, warp holding some of this rank's rows)
    mbar_init(red_full, (uint32_t)((split > 1 ? split - 1 : 1) * (split > 4 ? 1 : 4 / split)));
    *abort_flag = 0;
    fence_mbar_init();
    if (kADependent || kBDependent) {
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        if (kADependent) issue_a(kt_begin + i, i, pol_act);
        if (kBDependent) issue_b(kt_begin + i, i, pol_act);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // rank 0's reduction barrier must be initialized before any rank arrives on it
  if (split > 1) cluster_arrive_relaxed();

  if (warp == 0) {
    // ------------------------------------------- remaining stages (ring reuse)
    if (lane == 0 && nk > kStages) {
      int s = 0;
      uint32_t ph = 1;  // the prologue filled round 0 of every slot
      for (int64_t kt = kt_begin + kStages; kt < kt_end; ++kt) {
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&full[s], stage_bytes());
        issue_a(kt, s, kMode == kImagePlain ? pol_act : pol_weights);
        if (!C::kFused) issue_b(kt, s, kMode == kImageSwap ? pol_act : pol_weights);
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      // let copies already in flight land before the CTA exits
      for (int t = 0; t < kStages && t < nk; ++t) {
        const int64_t last_use = (nk - 1 - t) / kStages;  // round of the last copy into slot t
        wait_bounded(&full[t], (uint32_t)(last_use & 1), abort_flag, kDrainLimitCycles);
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
          for (int h = 0; h < C::kBTiles; ++h)
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

  if constexpr (C::kFused) {
    // ---------------------------------------- activation quantizers (warps 2-7)
    // The bf16 loads for up to kStages K tiles are in flight at once (a
    // register ring indexed at compile time), so DRAM latency is paid once,
    // not once per tile.
    if (warp >= 2) {
      constexpr int kRowsPerWarp = (BN + kQuantWarps - 1) / kQuantWarps;
      const int qw = warp - 2;
      uint4 w[kStages][kRowsPerWarp];
      auto load_tile = [&](int64_t kt, uint4 (&dst)[kRowsPerWarp]) {
        const int64_t col = kt * kTileK + lane * 8;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const int row = qw + i * kQuantWarps;
          dst[i] = (kt < kt_end && row < args.m && col < args.k) ? ldg_nc_v4(args.act + row * args.lda + col)
                                                                 : make_uint4(0, 0, 0, 0);
        }
      };
#pragma unroll
      for (int u = 0; u < kStages; ++u) load_tile(kt_begin + u, w[u]);
      uint32_t ph = 0;
      bool aborted = false;
      for (int64_t kt0 = kt_begin; kt0 < kt_end && !aborted; kt0 += kStages) {
#pragma unroll
        for (int u = 0; u < kStages; ++u) {
          const int64_t kt = kt0 + u;
          if (kt >= kt_end || aborted) continue;
          const bool slot_free = wait_bounded(&empty[u], ph ^ 1, abort_flag);
          if (!__all_sync(0xFFFFFFFFu, slot_free)) {  // keep the warp's decision uniform
            aborted = true;
            continue;
          }
          uint8_t* bd = smem + C::kOffBData + u * C::kBDataBytes;
          uint8_t* bsf = smem + C::kOffBSf + u * C::kBSfBytes;
#pragma unroll
          for (int i = 0; i < kRowsPerWarp; ++i) {
            const int row = qw + i * kQuantWarps;
            if (row < BN) {  // uniform across the warp
              uint32_t sbyte;
              const uint32_t packed = quantize_lane<kUseHardwareCvt>(w[u][i], sbyte);
              *reinterpret_cast<uint32_t*>(bd + tile_data_offset(row, lane * 4)) = packed;
              if ((lane & 3) == 0) bsf[tile_sf_offset(row, lane >> 2)] = (uint8_t)sbyte;
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&full[u]);
          load_tile(kt + kStages, w[u]);  // refill this slot of the ring
        }
        ph ^= 1;
      }
    }
  }

  // ------------------------------------------------------------- epilogue
  //   red: [S][128/S][kRedStride] fp32 rows this rank owns, pushed by rank q
  //        into slot q (a split cluster);
  //   stg: bf16 output tile, [BN][128] (swap-AB: rows are C rows) or
  //        [128][BN+8], in the stage buffers, idle once the accumulator is done.
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(smem);
  const int rows_per_rank = kTileRows / split;
  const int row_lo = rank * rows_per_rank, row_hi = row_lo + rows_per_rank;  // rows this CTA stores
  __syncwarp();
  if (split > 1) cluster_wait();  // every rank's barriers are initialized
  if (warp >= 2 && warp < 6) {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // accumulator row = tensor-memory lane
    const int owner = row / rows_per_rank;  // a warp's rows span two owners when each owns 16
    const bool ok = wait_bounded(accum, 0, abort_flag);
    tc_fence_after();
    // split: every row goes to slot `rank` of its owner's partial buffer (the
    // owner's own rows through the same path, to its own shared memory)
    const uint32_t dst =
        split > 1 ? map_cluster(smem_addr(red + (size_t)(rank * rows_per_rank + (row - owner * rows_per_rank)) *
                                                     C::kRedStride),
                                (uint32_t)owner)
                  : 0u;
    constexpr int kChunk = BN >= 32 ? 32 : 16;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += kChunk) {
      uint32_t r[kChunk];
      if constexpr (kChunk == 32) {
        tmem_load_32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, r);
      } else {
        tmem_load_16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, r);
      }
      tmem_load_wait();
      if (!ok) continue;
      if (split > 1) {
#pragma unroll
        for (int j = 0; j < kChunk; j += 4)
          st_cluster_f4(dst + (uint32_t)(c0 + j) * 4u,
                        make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                    __uint_as_float(r[j + 3])));
      } else if (C::kSwap) {
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          stg[(c0 + j) * C::kStgPitch + row] = __float2bfloat16_rn(__uint_as_float(r[j]));
      } else {
#pragma unroll
        for (int j = 0; j < kChunk; j += 8) {
          uint4 u;
          u.x = bf16x2_bits(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
          u.y = bf16x2_bits(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
          u.z = bf16x2_bits(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
          u.w = bf16x2_bits(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
          *reinterpret_cast<uint4*>(stg + row * C::kStgPitch + c0 + j) = u;
        }
      }
    }
    if (split > 1) {
      // The warp's pushes happen before the cluster-scope release of lane 0
      // (and of lane 16, when the warp's rows span two owners): one arrival
      // per warp and remote owner.
      __syncwarp();
      const bool first_of_owner = lane == 0 || (rows_per_rank < 32 && lane == 16);
      if (first_of_owner && owner != rank) mbar_arrive_remote(map_cluster(smem_addr(red_full), (uint32_t)owner));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {  // the accumulator has been read out
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }

  if (split > 1) {
    // ------------------------- sum this rank's rows over the S partials, in rank order
    wait_bounded_cluster(red_full, 0, abort_flag);  // the other ranks' rows have landed
    constexpr int kC4 = BN / 4;
    for (int g = threadIdx.x; g < rows_per_rank * kC4; g += C::kThreads) {
      const int rr = g % rows_per_rank, c4 = g / rows_per_rank;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < split; ++q) {
        const float4 v =
            *reinterpret_cast<const float4*>(red + (size_t)(q * rows_per_rank + rr) * C::kRedStride + c4 * 4);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const int row = row_lo + rr;
      if (C::kSwap) {
        stg[(c4 * 4 + 0) * C::kStgPitch + row] = __float2bfloat16_rn(acc.x);
        stg[(c4 * 4 + 1) * C::kStgPitch + row] = __float2bfloat16_rn(acc.y);
        stg[(c4 * 4 + 2) * C::kStgPitch + row] = __float2bfloat16_rn(acc.z);
        stg[(c4 * 4 + 3) * C::kStgPitch + row] = __float2bfloat16_rn(acc.w);
      } else {
        uint2 u;
        u.x = bf16x2_bits(acc.x, acc.y);
        u.y = bf16x2_bits(acc.z, acc.w);
        *reinterpret_cast<uint2*>(stg + row * C::kStgPitch + c4 * 4) = u;
      }
    }
    __syncthreads();
  }

  // ------------------------------------------ coalesced 16-byte stores of C
  if (C::kSwap) {
    // stg row j = C row j; stg column r = C column a_tile*128 + r
    const int64_t n0 = a_tile * kTileRows + row_lo;
    const int jmax = (int)(args.m < BN ? args.m : BN);
    const int nch = rows_per_rank / 8;
    for (int idx = threadIdx.x; idx < jmax * nch; idx += C::kThreads) {
      const int j = idx / nch, ch = idx % nch;
      const int64_t n = n0 + ch * 8;
      const __nv_bfloat16* src = stg + j * C::kStgPitch + row_lo + ch * 8;
      __nv_bfloat16* dst = args.c + j * args.ldc + n;
      if (n + 8 <= args.n) {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
      } else {
        for (int e = 0; e < 8 && n + e < args.n; ++e) dst[e] = src[e];
      }
    }
  } else {
    const int64_t m0 = a_tile * kTileRows;
    const int64_t n0 = b_tile * BN;
    constexpr int nch = BN / 8;
    for (int idx = threadIdx.x; idx < rows_per_rank * nch; idx += C::kThreads) {
      const int r = row_lo + idx / nch, ch = idx % nch;
      const int64_t mi = m0 + r;
      const int64_t n = n0 + ch * 8;
      if (mi >= args.m || n >= args.n) continue;
      const __nv_bfloat16* src = stg + r * C::kStgPitch + ch * 8;
      __nv_bfloat16* dst = args.c + mi * args.ldc + n;
      if (n + 8 <= args.n) {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
      } else {
        for (int e = 0; e < 8 && n + e < args.n; ++e) dst[e] = src[e];
      }
    }
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

// MXFP4_SPLIT_K=<1|2|4|8> overrides the K-split factor the planner picks
// (clamped to what the shape and the kernel allow); for tests and tuning.
static int split_override() {
  const char* v = getenv("MXFP4_SPLIT_K");
  if (!v) return 0;
  const int s = atoi(v);
  return (s == 1 || s == 2 || s == 4 || s == 8) ? s : 0;
}

int make_gemm_plan(int64_t m, int64_t n, int64_t k, GemmPlan* plan) {
  const int sms = num_sms();
  const int forced = split_override();
  const int64_t KT = ceil_div(k, kTileK);
  GemmPlan p{};
  if (m <= 128) {
    p.swap_ab = true;
    p.mode = m <= 32 ? kFusedSwap : kImageSwap;
    p.bn = m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 128;
    p.grid_x = ceil_div(n, kTileRows);
    const int s_max = 8;  // the kernels' kMaxSplit
    int s = 1;
    while (s < s_max && p.grid_x * s * 2 <= sms && KT / (s * 2) >= 1) s *= 2;
    if (forced) s = forced <= KT ? forced : 1;
    p.split = s;
    p.grid_y = s;
    p.workspace = p.mode == kFusedSwap ? 0 : (size_t)image_bytes(m, k);
  } else {
    p.swap_ab = false;
    p.mode = kImagePlain;
    const int64_t mt = ceil_div(m, kTileRows);
    p.bn = (mt * ceil_div(n, 256) >= sms) ? 256 : 128;
    p.grid_x = mt;
    const int64_t nt = ceil_div(n, p.bn);
    const int s_max = p.bn == 256 ? 1 : 8;  // the kernels' kMaxSplit
    int s = 1;
    while (s < s_max && mt * nt * s * 2 <= sms && KT / (s * 2) >= 2) s *= 2;
    if (forced) s = (forced <= KT && forced <= s_max) ? forced : 1;
    p.split = s;
    p.grid_y = nt * s;
    p.workspace = (size_t)image_bytes(m, k);
  }
  if (p.grid_x > 0x7FFFFFFF || p.grid_y > 65535) return 1;
  *plan = p;
  return 0;
}

template <int BN, int kMode>
static cudaError_t launch_one(const GemmPlan& plan, const GemmArgs& args, cudaStream_t stream) {
  using C = Cfg<BN, kMode>;
  if (plan.split > C::kMaxSplit) return cudaErrorInvalidConfiguration;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  if (kMode != kFusedSwap) {  // dependent of the quantization kernel
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN, kMode>, args);
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
  if (plan.mode == kFusedSwap) {
    args.a_img = static_cast<const uint8_t*>(b_image);
    args.a_rows = n;
    args.act = static_cast<const uint16_t*>(a_bf16);
    switch (plan.bn) {
      case 16: return launch_one<16, kFusedSwap>(plan, args, stream);
      case 32: return launch_one<32, kFusedSwap>(plan, args, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  cudaError_t e = launch_quant_image(a_bf16, m, k, lda, workspace, stream);
  if (e != cudaSuccess) return e;
  if (plan.mode == kImageSwap) {
    args.a_img = static_cast<const uint8_t*>(b_image);
    args.a_rows = n;
    args.b_img = static_cast<const uint8_t*>(workspace);
    args.b_rows = m;
    switch (plan.bn) {
      case 64: return launch_one<64, kImageSwap>(plan, args, stream);
      case 128: return launch_one<128, kImageSwap>(plan, args, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  args.a_img = static_cast<const uint8_t*>(workspace);
  args.a_rows = m;
  args.b_img = static_cast<const uint8_t*>(b_image);
  args.b_rows = n;
  switch (plan.bn) {
    case 128: return launch_one<128, kImagePlain>(plan, args, stream);
    case 256: return launch_one<256, kImagePlain>(plan, args, stream);
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
