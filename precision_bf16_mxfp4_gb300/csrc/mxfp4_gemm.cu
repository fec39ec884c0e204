// MXFP4 GEMM  C[m,n] = quant(A) . B^T  on tcgen05 block-scaled tensor cores.
//
// Semantics (kernelbot amd-mxfp4-mm pages, submission 752099: the
// `tl.dot_scaled(a, a_scale, "e2m1", b, b_scale, "e2m1", acc)` product with
// fp32 accumulation and a bf16 result; submission 694791 for the quantizer):
//   C[i,j] = bf16( sum_kb 2^(sa[i,kb]-127) 2^(sb[j,kb]-127) sum_t a[i,32kb+t] b[j,32kb+t] )
//
// One CTA computes a 128 x BN accumulator tile in tensor memory.  The MMA's
// 128-row operand ("MMA-A") comes from a tiled operand image (see
// mxfp4_device.cuh) through bulk copies.  Modes:
//   kFusedSwap (m <= 32): swap-AB.  MMA-A = prepacked weights (n on the
//     128-row side); MMA-B = the activations, quantized by producer warps
//     from bf16 straight into shared memory in the MMA operand and scale
//     layouts, so quantized A never reaches HBM.  BN = m padded to 16/32.
//   kImageSwap (32 < m <= 128): swap-AB; MMA-B = the first BN rows of the
//     activation image that quant_image_kernel wrote into the workspace.
//   kImagePlain (m > 128, few tiles): MMA-A = activation image, MMA-B = 128
//     weight rows.  With at least one 128 x 256 tile per SM the CTA-pair
//     kernel below takes over (256 x 256 tiles, tcgen05 cta_group::2).
// In the image modes the GEMM is launched as a programmatic dependent of the
// quantization kernel: it streams its first weight stages at once and waits
// for the activation image only before loading it.
//
// Pipeline stages hold kSuperK consecutive K blocks (256 K each) of every
// operand row tile, so each stage is one bulk copy per row tile: the TMA
// engine's throughput per SM grows with the size of each copy (about
// 40 GB/s for 16 KiB copies, 120-160 GB/s for 48-64 KiB ones, measured on
// GB300), not with the number of copies in flight.  Each operand stream has
// its own issuing thread; the weights' first round goes out from thread 0
// before anything else.
//
// K may be split across the S CTAs (1 <= S <= 8) of a thread-block cluster.
// Rank r owns accumulator rows [floor(128r/S), floor(128(r+1)/S)) (the ranks
// own 128/S rows each, give or take one): every rank gathers the rows of its
// fp32 partial per owner in shared memory (its own rows straight into its
// slot) and sends each owner its rows as one DSMEM bulk copy into slot r of
// the owner's reduction buffer, completing on the owner's mbarrier; the owner
// adds the S slots in rank order (deterministic) and stores its rows.
//
// Warp roles: warp 0 issues the weights' bulk copies (the last warp, in the
// image modes, the activation image's); warp 1 owns tensor memory and issues
// the MMAs (one thread); warps 2-5 write each stage's scale factors into
// tensor memory (tcgen05.st) and drain the accumulator; in kFusedSwap warps
// 2-9 quantize the activations and write the scales, and warps 6-9 also drain
// the accumulator when BN = 32.  Every wait is bounded: a wait that runs out
// sets a device flag and the CTA winds down.
#include <cuda.h>  // CUtensorMap (a type only: the library links no driver symbol)
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
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
constexpr int kSuperK = 2;                          // K blocks per pipeline stage

enum GemmMode : int { kFusedSwap = 0, kImageSwap = 1, kImagePlain = 2 };

struct GemmArgs {
  const uint8_t* a_img;  // MMA-A operand image
  const uint8_t* b_img;  // MMA-B operand image (image modes)
  int64_t b_rows;        // rows of the matrix in b_img
  const uint16_t* act;   // bf16 activations (kFusedSwap)
  int64_t lda;
  int64_t m, n, k;
  int64_t kt_count;  // K blocks of 256
  __nv_bfloat16* c;
  int64_t ldc;
  int split;
  int drop_copies;  // test hook: the MMA issuer's operand wait runs out (see launch_gemm)
};

template <int BN, int kMode>
struct Cfg {
  static constexpr bool kFused = kMode == kFusedSwap;
  static constexpr bool kSwap = kMode != kImagePlain;
  // warps: 0 issues the weights' bulk copies (in the image modes the last
  // warp issues the activation image's), 1 issues MMAs, 2-5 write the scale
  // factors to tensor memory and drain the accumulator.  kFusedSwap: warps
  // 2-9 quantize A, one thread per (row, 32-element block) of a K block;
  // BN = 16 needs only half of them per K block, so the threads form
  // kQuantGroups groups that take the stage's K blocks in turn; thread 0
  // issues the weights' first round at setup, warp 0 the later stages
  static constexpr int kQuantWarps = kFused ? 8 : 0;
  static constexpr int kQuantGroups = kFused ? 32 / BN : 1;
  // K blocks in a quantizer thread's register ring: two stages' worth for
  // BN = 32, three stages (one block each) for BN = 16, within the 168
  // registers a thread of a 10-warp CTA can have
  static constexpr int kRing = BN >= 32 ? 2 * kSuperK : 3;
  static constexpr int kEpiWarps = (kFused && BN >= 32) ? 8 : 4;  // accumulator-draining warps (from warp 2)
  static constexpr int kEpiCols = BN / (kEpiWarps / 4);         // accumulator columns per draining warp
  static constexpr int kThreads = kFused ? 32 * (2 + kQuantWarps) : 32 * 7;
  static constexpr int kActProducerWarp = kFused ? 0 : kThreads / 32 - 1;  // issues the activation stream
  static constexpr int kBRows = BN;                                    // MMA N (<= 128 here)
  // stages in the ring: kFusedSwap keeps four in flight (a thin CTA's whole
  // K range for k <= 2048, or a split rank's share), the image modes three
  static constexpr int kStages = kFused ? 4 : 3;
  static constexpr int kABytes = kSuperK * kTileBytes;                 // MMA-A bytes per stage
  static constexpr int kBBlock = kFused ? BN * 128 + kTileSfBytes : kTileBytes;  // per K block
  static constexpr int kBSfOffset = kFused ? BN * 128 : kTileDataBytes;          // scales inside a B block
  static constexpr int kBBytes = kSuperK * kBBlock;                    // MMA-B bytes per stage
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffBars = kOffB + kStages * kBBytes;
  static constexpr int kOffMisc = kOffBars + (4 * kStages + 2) * 8;
  // Once this CTA's accumulator is complete its stage buffers are idle and
  // hold the bf16 output tile (kImagePlain) and the split-K rows other ranks
  // own, gathered per owner.  The partials of the rows this rank owns
  // ([S][128/S][kRedStride], slot q written by rank q) get a region of their
  // own in kFusedSwap, so a fast rank can send while this one still runs its
  // MMAs; the image modes need that shared memory for their third stage and
  // keep them in the stage buffers too, sending only after a cluster barrier
  // that follows every rank's accumulator.
  static constexpr int kMaxSplit = 8;
  static constexpr int kRedStride = BN + 4;               // fp32 partial-row pitch (floats)
  // S slots of up to ceil(128 / S) rows each: at most 128 + S - 1 rows
  static constexpr int kRedBytes = (128 + kMaxSplit - 1) * kRedStride * 4;
  static constexpr bool kRedInStages = !kFused;
  static constexpr int kStgPitch = BN + 8;                // elements (kImagePlain)
  static constexpr int kStgBytes = kSwap ? 0 : 128 * kStgPitch * 2;
  static constexpr int kOffOut = (kStgBytes + 1023) & ~1023;
  static constexpr int kOffRed = kRedInStages ? kOffOut + ((kRedBytes + 1023) & ~1023) : (kOffMisc + 16 + 15) & ~15;
  static_assert(kOffOut + kRedBytes <= kOffBars, "the gather buffer must fit in the stage buffers");
  static_assert(!kSwap || BN * (kTileRows + 8) * 2 <= kOffBars, "the swap-AB output rows must fit in the stage buffers");
  static_assert(!kRedInStages || kOffRed + kRedBytes <= kOffBars, "epilogue buffers must fit in the stage buffers");
  static constexpr int kSmemBytes = (kRedInStages ? kOffMisc + 16 : kOffRed + kRedBytes) + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kBBlock % 1024 == 0, "swizzled operand blocks must stay 1024-byte aligned");
  // tensor memory: accumulator columns, then per-stage scale-factor columns
  // (8 per K block for A, 8 per K block for B)
  static constexpr int kAccCols = BN;
  static constexpr int kSfColsPerStage = kSuperK * 16;
  static constexpr int kTmemNeed = kAccCols + kStages * kSfColsPerStage;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "tensor memory");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "MMA N");
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

// Winding down after a timeout: wait up to kDrainLimitCycles for a phase
// (the bulk copies this CTA issued must land before it exits), whatever the
// abort flag says.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kDrainLimitCycles) {
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

// Same, polling with test_wait (for waits on arrivals from the other CTA of
// a pair, which a suspended try_wait notices late).
__device__ __forceinline__ bool wait_bounded_poll(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait_cluster(bar, parity)) return true;
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

// Scale factors of one K block (two 512-byte atoms in shared memory) into 8
// tensor-memory columns of the calling warp's 32-lane quadrant, with the
// column contents tcgen05.cp.32x128b.warpx4 would produce: lane l holds the
// 16 bytes of atom row l (row groups l, l+32, l+64, l+96; K blocks 0-3) in 4
// columns and the second atom's 16 bytes (K blocks 4-7) in the next 4.
// Measured on GB300, a tcgen05.cp stalls the MMA queue for hundreds of
// cycles; these stores run on warps other than the MMA issuer.
__device__ __forceinline__ void store_block_scales(uint32_t taddr, const uint8_t* sf_smem, int lane) {
  const uint4 lo = *reinterpret_cast<const uint4*>(sf_smem + lane * 16);
  const uint4 hi = *reinterpret_cast<const uint4*>(sf_smem + kAtomBytes + lane * 16);
  const uint32_t v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  tmem_store_8(taddr, v);
}

// Accumulator rows of a K split over `split` ranks: rank q owns rows
// [split_row0(q), split_row0(q + 1)); owner_of(r) is the rank that owns row r.
__device__ __forceinline__ int split_row0(int q, int split) { return q * kTileRows / split; }
__device__ __forceinline__ int owner_of(int r, int split) { return ((r + 1) * split - 1) / kTileRows; }

// K steps of 64 in the K block starting at element kt * 256
__device__ __forceinline__ int k_steps(int64_t k, int64_t kt) {
  const int64_t rem = k - kt * kTileK;
  return rem >= kTileK ? 4 : (int)ceil_div(rem, 64);
}

template <int BN, int kMode>
__global__ void __launch_bounds__(Cfg<BN, kMode>::kThreads, 1) gemm_kernel(const GemmArgs args) {
  using C = Cfg<BN, kMode>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* empty = full + C::kStages;
  uint64_t* accum = empty + C::kStages;
  uint64_t* red_full = accum + 1;  // the other ranks' partial rows owned by this rank have landed
  uint64_t* act_ready = red_full + 1;      // kFusedSwap: the stage's activations are quantized
  uint64_t* sf_ready = act_ready + C::kStages;  // the stage's scale factors are in tensor memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = args.split;
  const int rank = split > 1 ? (int)(blockIdx.y % split) : 0;
  const int64_t a_tile = blockIdx.x;
  const int64_t b_tile = blockIdx.y / split;  // row tile of the MMA-B image (plain mode)
  const int64_t KT = args.kt_count;
  const int64_t kt_begin = KT * rank / split;
  const int64_t kt_end = KT * (rank + 1) / split;
  const int nss = (int)ceil_div(kt_end - kt_begin, kSuperK);  // pipeline stages this CTA runs

  // kFusedSwap: the quantizer threads start loading their bf16 blocks for
  // the first C::kRing K blocks right away, before any setup: DRAM latency is
  // the long pole.  Ring position u holds K block kt0 + u (block u % kSuperK
  // of its stage); the register ring is indexed at compile time.  Quantizer
  // thread qt owns row qt / 8 and 32-element block qt % 8 of every K block.
  const bool quantizer = C::kFused && warp >= 2 && warp < 2 + C::kQuantWarps;
  const int qt = (int)threadIdx.x - 64;
  const int q_row = (qt % (BN * 8)) >> 3, q_blk = qt & 7;
  const int q_group = qt / (BN * 8);  // K block q_group + p * kQuantGroups of every stage
  uint4 w[C::kRing][4];
  auto load_block = [&](int64_t kt, uint4 (&dst)[4]) {
    const int64_t col = kt * kTileK + q_blk * 32;
    if (kt < kt_end && q_row < args.m && col < args.k) {
      ldg_nc_block(args.act + q_row * args.lda + col, dst);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(0, 0, 0, 0);
    }
  };
  // a thread's ring: kRingStages stages of kPerStage K blocks
  constexpr int kPerStage = kSuperK / C::kQuantGroups;
  constexpr int kRingStages = C::kRing / kPerStage;
  static_assert(kSuperK % C::kQuantGroups == 0 && C::kRing % kPerStage == 0, "quantizer ring shape");
  auto ring_kt = [&](int ss, int p) -> int64_t {  // K block of the thread's p-th block in stage ss
    return kt_begin + (int64_t)ss * kSuperK + q_group + p * C::kQuantGroups;
  };
  if (quantizer) {
#pragma unroll
    for (int u = 0; u < C::kRing; ++u) load_block(ring_kt(u / kPerStage, u % kPerStage), w[u]);
  }

  const bool b_valid = !C::kFused && b_tile < ceil_div(args.b_rows, kTileRows);
  auto stage_kblocks = [&](int ss) -> int {
    const int64_t left = kt_end - (kt_begin + (int64_t)ss * kSuperK);
    return left < kSuperK ? (int)left : kSuperK;
  };
  auto issue_a = [&](int ss, int s, uint64_t policy) {
    const int64_t kt0 = kt_begin + (int64_t)ss * kSuperK;
    const uint32_t bytes = (uint32_t)stage_kblocks(ss) * kTileBytes;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_load_hint(smem + C::kOffA + s * C::kABytes, args.a_img + image_block(a_tile, kt0, KT), bytes, &full[s],
                   policy);
  };
  auto issue_b = [&](int ss, int s, uint64_t policy) {
    if (!b_valid) {  // a weight row tile beyond n: nothing to copy
      mbar_arrive(&full[s]);
      return;
    }
    const int64_t kt0 = kt_begin + (int64_t)ss * kSuperK;
    const int cnt = stage_kblocks(ss);
    if (kMode == kImageSwap && BN < kTileRows) {
      // the MMA reads only the first BN rows of each activation block: copy
      // those rows' data and the block's scale atoms, not the whole block
      mbar_arrive_expect_tx(&full[s], (uint32_t)cnt * (BN * 128 + kTileSfBytes));
      for (int j = 0; j < cnt; ++j) {
        const uint8_t* src = args.b_img + image_block(b_tile, kt0 + j, KT);
        uint8_t* dst = smem + C::kOffB + s * C::kBBytes + j * C::kBBlock;
        bulk_load_hint(dst, src, BN * 128, &full[s], policy);
        bulk_load_hint(dst + kTileDataBytes, src + kTileDataBytes, kTileSfBytes, &full[s], policy);
      }
      return;
    }
    const uint32_t bytes = (uint32_t)cnt * kTileBytes;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_load_hint(smem + C::kOffB + s * C::kBBytes, args.b_img + image_block(b_tile, kt0, KT), bytes, &full[s],
                   policy);
  };
  // Two operand streams: W, the weights, and (image modes) X, the activation
  // image the preceding quantization kernel writes.  Each has one issuing
  // thread (the bulk copies one thread issues are serialized) and arrives on
  // a stage's full barrier once, with its bytes.
  constexpr bool kWIsA = kMode != kImagePlain;
  auto issue_w = [&](int ss, int s) {
    if (kWIsA) issue_a(ss, s, policy_evict_first());
    else issue_b(ss, s, policy_evict_first());
  };
  auto issue_x = [&](int ss, int s) {
    if (kWIsA) issue_b(ss, s, policy_evict_last());
    else issue_a(ss, s, policy_evict_last());
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], C::kFused ? 1 : 2);  // one arrival (with its bytes) per operand stream
      if (C::kFused) mbar_init(&act_ready[s], C::kQuantWarps * 32);  // every quantizer thread
      mbar_init(&sf_ready[s], C::kFused ? 8 : 4);  // one arrival per scale-factor warp
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    // the other ranks' partial rows arrive as bulk copies: one arrival (this
    // thread's, below) plus their bytes
    mbar_init(red_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (split > 1)
      mbar_arrive_expect_tx(red_full, (uint32_t)((split - 1) * (split_row0(rank + 1, split) - split_row0(rank, split)) *
                                                 C::kRedStride * 4));
    if (!args.drop_copies) {
      // The weight stream is the long pole: its whole first round starts
      // now, before the tensor-memory allocation and the setup barrier (on
      // GB300 this measured ~0.4 us faster at m = 16, k = 7168 than issuing
      // stages 1.. from other warps after the barrier).
      const int pre = nss < C::kStages ? nss : C::kStages;
      for (int i = 0; i < pre; ++i) issue_w(i, i);
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
  // the owners' reduction barriers must be initialized before any rank arrives on them
  if (split > 1) cluster_arrive_relaxed();

  if (warp == 0 || warp == C::kActProducerWarp) {
    // ------------------------------------------------ bulk-copy producers
    // warp 0: the weight stream's later rounds; the last warp (image modes):
    // the activation stream, after the quantization kernel has finished
    if (lane == 0 && !args.drop_copies) {
      const bool x_stream = !C::kFused && warp == C::kActProducerWarp;
      if (x_stream) pdl_wait();
      int issued = x_stream ? 0 : (nss < C::kStages ? nss : C::kStages);  // the weights' first round went out at setup
      for (int ss = issued; ss < nss; ++ss) {
        const int s = ss % C::kStages;
        if (ss >= C::kStages && !wait_bounded(&empty[s], (uint32_t)(((ss / C::kStages) & 1) ^ 1), abort_flag)) break;
        if (x_stream) issue_x(ss, s);
        else issue_w(ss, s);
        issued = ss + 1;
      }
      if (*abort_flag) {  // let the copies in flight land before the CTA exits
        for (int t = 0; t < C::kStages && t < issued; ++t) {
          const int last = t + ((issued - 1 - t) / C::kStages) * C::kStages;
          drain_wait(&full[t], (uint32_t)((last / C::kStages) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool accumulate = false;
      for (int ss = 0; ss < nss; ++ss) {
        const int s = ss % C::kStages;
        const uint32_t ph = (uint32_t)((ss / C::kStages) & 1);
        if (!wait_bounded(&full[s], ph, abort_flag) || !wait_bounded(&sf_ready[s], ph, abort_flag)) break;
        tc_fence_after();
        const uint32_t sfa = tmem + C::kAccCols + s * C::kSfColsPerStage;
        const uint32_t sfb = sfa + kSuperK * 8;
        const int cnt = stage_kblocks(ss);
        const int64_t kt0 = kt_begin + (int64_t)ss * kSuperK;
        // One thread issues every MMA, so per-MMA address arithmetic sits on
        // the critical path: the descriptors are built once per stage and
        // advanced in their start-address field (byte offset / 16; shared
        // addresses stay below 256 KiB, so the 14-bit field cannot carry).
        const uint64_t a_desc = smem_desc(smem_addr(smem + C::kOffA + s * C::kABytes), 0, 1024, kLayoutSwizzle128);
        const uint64_t b_desc = smem_desc(smem_addr(smem + C::kOffB + s * C::kBBytes), 0, 1024, kLayoutSwizzle128);
        auto issue = [&](int j, int kk) {
          // scale-factor id (2 per 64-K step) selects the byte of the 4-byte group
          constexpr uint32_t kIdEven = idesc_mxf4(128, C::kBRows, 0, 0), kIdOdd = idesc_mxf4(128, C::kBRows, 2, 2);
          mma_mxf4(tmem, a_desc + (uint64_t)((j * kTileBytes + kk * 32) >> 4),
                   b_desc + (uint64_t)((j * C::kBBlock + kk * 32) >> 4), (kk & 1) ? kIdOdd : kIdEven,
                   sfa + j * 8 + (kk >> 1) * 4, sfb + j * 8 + (kk >> 1) * 4, accumulate ? 1u : 0u);
          accumulate = true;
        };
        // a whole K block's four MMAs go out from one asm block; a K tail of
        // 64-element steps one MMA at a time
        auto kblock = [&](int j) {
          constexpr uint32_t kIdEven = idesc_mxf4(128, C::kBRows, 0, 0), kIdOdd = idesc_mxf4(128, C::kBRows, 2, 2);
          mma_mxf4_kblock(tmem, a_desc + (uint64_t)((j * kTileBytes) >> 4),
                          b_desc + (uint64_t)((j * C::kBBlock) >> 4), kIdEven, kIdOdd, sfa + j * 8, sfb + j * 8,
                          accumulate ? 1u : 0u);
          accumulate = true;
        };
        if (cnt == kSuperK && (kt0 + kSuperK) * kTileK <= args.k) {  // whole stage
#pragma unroll
          for (int j = 0; j < kSuperK; ++j) kblock(j);
        } else {  // last stage: fewer K blocks, or a K tail
          for (int j = 0; j < cnt; ++j) {
            const int steps = k_steps(args.k, kt0 + j);
            if (steps == 4) {
              kblock(j);
            } else {
              for (int kk = 0; kk < steps; ++kk) issue(j, kk);
            }
          }
        }
        mma_commit(&empty[s]);
      }
      mma_commit(accum);  // fires once every MMA above has completed
    }
    __syncwarp();
  }

  // Scale factors of stage ss into tensor memory by a warp per 32-lane
  // quadrant (the warp's own, warp % 4): the MMA-A scales once the stage's
  // copies have landed, the MMA-B scales (kFusedSwap: once every quantizer
  // thread has finished the stage); then the MMA thread may issue the stage's
  // MMAs.  Image modes: warps 2-5 write both.  kFusedSwap: warps 6-9 write the
  // MMA-A (weight) scales and warps 2-5 the MMA-B (activation) scales.
  auto write_stage_scales = [&](int ss, bool do_a, bool do_b) -> bool {
    const int s = ss % C::kStages;
    const uint32_t ph = (uint32_t)((ss / C::kStages) & 1);
    const uint32_t quad_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t sfa = quad_base + C::kAccCols + s * C::kSfColsPerStage;
    const uint32_t sfb = sfa + kSuperK * 8;
    const int cnt = stage_kblocks(ss);
    if (do_a) {
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(&full[s], ph, abort_flag))) return false;
      for (int j = 0; j < cnt; ++j)
        store_block_scales(sfa + j * 8, smem + C::kOffA + s * C::kABytes + j * kTileBytes + kTileDataBytes, lane);
    }
    if (do_b) {
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(C::kFused ? &act_ready[s] : &full[s], ph, abort_flag))) return false;
      for (int j = 0; j < cnt; ++j)
        store_block_scales(sfb + j * 8, smem + C::kOffB + s * C::kBBytes + j * C::kBBlock + C::kBSfOffset, lane);
    }
    tmem_store_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sf_ready[s]);
    return true;
  };

  if constexpr (C::kFused) {
    // ------------------------------------- activation quantizers (warps 2-9)
    if (quantizer) {
      bool aborted = false;
      for (int ss0 = 0; ss0 < nss && !aborted; ss0 += kRingStages) {
#pragma unroll
        for (int rs = 0; rs < kRingStages; ++rs) {
          const int ss = ss0 + rs;
          if (ss >= nss || aborted) continue;
          const int s = ss % C::kStages;
          const bool slot_free = wait_bounded(&empty[s], (uint32_t)(((ss / C::kStages) & 1) ^ 1), abort_flag);
          if (!__all_sync(0xFFFFFFFFu, slot_free)) {  // keep the warp's decision uniform
            aborted = true;
            continue;
          }
          const int cnt = stage_kblocks(ss);
#pragma unroll
          for (int p = 0; p < kPerStage; ++p) {
            const int u = rs * kPerStage + p, j = q_group + p * C::kQuantGroups;
            if (j < cnt) {
              uint8_t* blk = smem + C::kOffB + s * C::kBBytes + j * C::kBBlock;
              uint32_t sbyte;
              const uint4 packed = quantize_block32<kUseHardwareCvt>(w[u], sbyte);
              *reinterpret_cast<uint4*>(blk + tile_data_offset(q_row, q_blk * 16)) = packed;
              blk[C::kBSfOffset + tile_sf_offset(q_row, q_blk)] = (uint8_t)sbyte;
            }
            load_block(ring_kt(ss + kRingStages, p), w[u]);  // refill this ring position
          }
          // every quantizer thread arrives once per stage, with or without a block in it
          fence_proxy_async_smem();
          mbar_arrive(&act_ready[s]);
          // The quantizer warps also write the scales (2-5 activations, 6-9
          // weights), one stage behind their quantization: by then the other
          // quantizers have finished that stage and its weights have landed,
          // so neither role waits on the other.
          if (ss > 0 && !write_stage_scales(ss - 1, warp >= 6, warp < 6)) aborted = true;
        }
      }
      if (!aborted && nss > 0) write_stage_scales(nss - 1, warp >= 6, warp < 6);
    }
  } else {
    if (warp >= 2 && warp < 6) {
      for (int ss = 0; ss < nss; ++ss)
        if (!write_stage_scales(ss, true, true)) break;
    }
  }

  // ------------------------------------------------------------- epilogue
  //   red: [S][128/S][kRedStride] fp32 rows this rank owns, pushed by rank q
  //        into slot q (a split cluster);
  //   stg: bf16 output tile in the stage buffers, idle once the accumulator
  //        is done: [128][BN+8] (kImagePlain), or C's rows [BN][128+8]
  //        (swap-AB, unsplit).
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(smem);
  constexpr int kSwapPitch = kTileRows + 8;  // elements: 272-byte rows, 16-byte aligned
  const int slot_rows = (kTileRows + split - 1) / split;  // pitch of the per-owner slots (rows)
  const int row_lo = split_row0(rank, split);             // first accumulator row this CTA stores
  const int my_rows = split_row0(rank + 1, split) - row_lo;
  __syncwarp();
  if (split > 1) cluster_wait();  // every rank's barriers are initialized
  // Warps 2-5 drain the accumulator, warp w reading tensor-memory lane
  // quadrant w % 4; with 8 quantizer warps (kFusedSwap, BN = 32) warps 6-9
  // take the upper half of the same quadrants' columns, so each warp stores
  // half as many C rows.
  if (warp >= 2 && warp < 2 + C::kEpiWarps) {
    const int quad = warp & 3;
    const int col_lo = ((warp - 2) >> 2) * C::kEpiCols;
    const int row = quad * 32 + lane;  // accumulator row = tensor-memory lane
    const int owner = owner_of(row, split);  // a warp's rows can span two owners
    const bool ok = wait_bounded(accum, 0, abort_flag);
    tc_fence_after();
    // split: this rank's own rows go to its slot of `red`; the rows another
    // rank owns are gathered per owner in the (idle) stage buffers and sent
    // below as one bulk copy per owner
    float* part = (owner == rank ? red + (size_t)rank * slot_rows * C::kRedStride
                                 : reinterpret_cast<float*>(smem + C::kOffOut) + (size_t)owner * slot_rows * C::kRedStride) +
                  (size_t)(row - split_row0(owner, split)) * C::kRedStride;
    constexpr int kChunk = C::kEpiCols >= 32 ? 32 : 16;
#pragma unroll 1
    for (int c0 = col_lo; c0 < col_lo + C::kEpiCols; c0 += kChunk) {
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
          *reinterpret_cast<float4*>(part + c0 + j) = make_float4(
              __uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
      } else if (C::kSwap) {
        // accumulator row = C column n, accumulator column = C row: the
        // values go to shared memory as C rows (the warp's 32 lanes fill 32
        // consecutive columns of each row) and are stored below as 16-byte
        // pieces of whole rows
        __nv_bfloat16* p = stg + (size_t)c0 * kSwapPitch + row;
#pragma unroll
        for (int j = 0; j < kChunk; ++j) p[j * kSwapPitch] = __float2bfloat16_rn(__uint_as_float(r[j]));
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
    if (split > 1) fence_proxy_async_smem();  // the gathered rows are read by bulk copies
    if (C::kSwap && split == 1) {
      // C rows [0, min(m, BN)) of this tile's 128 columns from shared memory:
      // 16 lanes per 256-byte row, 16 bytes each (8 columns)
      named_barrier_sync(1, C::kEpiWarps * 32);
      const int64_t n0 = a_tile * kTileRows;
      const int rows = args.m < BN ? (int)args.m : BN;
      for (int idx = (int)threadIdx.x - 64; idx < rows * (kTileRows / 8); idx += C::kEpiWarps * 32) {
        const int mr = idx >> 4, ch = idx & 15;
        const int64_t n = n0 + ch * 8;
        if (!ok || n >= args.n) continue;
        const __nv_bfloat16* src = stg + (size_t)mr * kSwapPitch + ch * 8;
        __nv_bfloat16* dst = args.c + (int64_t)mr * args.ldc + n;
        if (n + 8 <= args.n) {
          *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
        } else {
          for (int e = 0; e < 8 && n + e < args.n; ++e) dst[e] = src[e];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {  // the accumulator has been read out
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }

  if (split > 1) {
    // --------------- reduce-scatter: slot `rank` of every other owner's `red`
    // (in the owners' stage buffers: every rank's accumulator must be complete)
    if (C::kRedInStages) cluster_sync();
    if (threadIdx.x == 0 && !*abort_flag) {
      for (int o = 0; o < split; ++o) {
        if (o == rank) continue;
        const uint32_t bytes = (uint32_t)((split_row0(o + 1, split) - split_row0(o, split)) * C::kRedStride * 4);
        bulk_copy_to_cluster(map_cluster(smem_addr(red + (size_t)rank * slot_rows * C::kRedStride), (uint32_t)o),
                             reinterpret_cast<const float*>(smem + C::kOffOut) + (size_t)o * slot_rows * C::kRedStride,
                             bytes, map_cluster(smem_addr(red_full), (uint32_t)o));
      }
      bulk_commit_group();
    }
    // ------------------------- sum this rank's rows over the S partials, in rank order
    wait_bounded_cluster(red_full, 0, abort_flag);  // the other ranks' rows have landed
    constexpr int kC4 = BN / 4;
    for (int g = threadIdx.x; g < my_rows * kC4; g += C::kThreads) {
      const int rr = g % my_rows, c4 = g / my_rows;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < split; ++q) {
        const float4 v =
            *reinterpret_cast<const float4*>(red + (size_t)(q * slot_rows + rr) * C::kRedStride + c4 * 4);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const int row = row_lo + rr;
      if (C::kSwap) {  // consecutive threads: consecutive C columns of C rows 4*c4 .. 4*c4+3
        const int64_t n = a_tile * kTileRows + row;
        const float v[4] = {acc.x, acc.y, acc.z, acc.w};
        if (n < args.n) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (c4 * 4 + e < args.m) args.c[(c4 * 4 + e) * args.ldc + n] = __float2bfloat16_rn(v[e]);
        }
      } else {
        uint2 u;
        u.x = bf16x2_bits(acc.x, acc.y);
        u.y = bf16x2_bits(acc.z, acc.w);
        *reinterpret_cast<uint2*>(stg + row * C::kStgPitch + c4 * 4) = u;
      }
    }
    if (!C::kSwap) __syncthreads();
  }

  // this CTA's outgoing bulk copies must have read their source before it exits
  if (split > 1 && threadIdx.x == 0) bulk_wait_group_read0();

  // ------------------------------------------ coalesced 16-byte stores of C
  // (swap-AB stores straight from registers above)
  if constexpr (!C::kSwap) {
    const int64_t m0 = a_tile * kTileRows;
    const int64_t n0 = b_tile * BN;
    constexpr int nch = BN / 8;
    for (int idx = threadIdx.x; idx < my_rows * nch; idx += C::kThreads) {
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


// ------------------------------------ CTA-pair persistent tile loop (m > 128, many tiles)
// When the output has at least one 128 x 256 tile per SM, the GEMM runs on
// CTA pairs (clusters of two): each pair computes 256 x 256 output tiles
// t = pair, pair + pairs, ... with 256 x 256 x 64 block-scaled MMAs
// (tcgen05 cta_group::2) that the even CTA issues.  Tiles are numbered
// along C's rows first (t -> row tile mt = t / tiles_n, column tile
// nt = t % tiles_n), so a wave of pairs needs a few activation row tiles and
// every weight tile: the weights are what the copies can fetch while the
// activation's quantization is still running, and this order measured 2.4 us
// faster at m = 4096, n = 7168, k = 2048 than walking the columns first
// (39.5 vs 41.9 us; the GEMM alone on a ready image is the same either way).
// CTA r of a pair holds
// activation row tile 2·mt + r and weight row tile 2·nt + r of every K block
// in its shared memory, and accumulator rows [128r, 128r + 128) in its tensor
// memory.  Per SM this halves the weight bytes that each MMA reads from
// shared memory and that the bulk copies write there, against a one-CTA
// 128 x 256 tile, and the freed space deepens the operand ring to three
// stages of two K blocks (the turnaround of a stage - MMAs done, refill
// issued, 68 KiB landed - is longer than two stages of MMAs on GB300).  The
// ring runs continuously across tiles.
//
// Hand-offs: a CTA's full[s] completes when its copies have landed and its
// scale warps - which write the stage's e8m0 atoms, read straight from the
// operand images, into their own CTA's tensor memory once the slot's
// previous MMAs have completed - have arrived, so the MMA thread polls one
// barrier per stage.  In the odd CTA a relay thread waits for that phase and
// makes one arrival on the even CTA's full[s].
// The MMA thread's commits arrive on empty[s] and acc_full in both CTAs
// (multicast).  The epilogue warps read their accumulator rows into
// registers and arrive on the even CTA's acc_empty; their global stores
// overlap the next tile's MMAs.  Only two kinds of thread-issued arrival
// cross between the CTAs - the relay's and the odd epilogue warps' - both
// relaxed (they publish nothing: the bytes and scales they report are in
// place, the accumulator reads they report have completed), and the threads
// that wait for them poll: on GB300 a cluster-scope release arrive stalls
// the issuing thread while the SM's global stores are in flight, and a
// suspended try_wait notices a remote arrival late.
//
// Warps: 0-7 epilogue (two per 32-lane quadrant, 128 columns each), 8-11
// scale factors, 12 activation copies (and setup), 13 tensor memory and MMA
// issue (the relay in the odd CTA), 14 weight copies.
struct PairCfg {
  static constexpr int BN = 256;     // output columns per pair tile (128 weight rows per CTA)
  static constexpr int kStages = 3;  // ring depth
  static constexpr int kSuperK = 2;  // K blocks per stage (one bulk copy per operand and stage)
  static constexpr int kThreads = 32 * 15;
  static constexpr int kStageOpBytes = kSuperK * kTileBytes;  // one operand, one stage
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kStages * kStageOpBytes;
  static constexpr int kOffStg = kOffB + kStages * kStageOpBytes;
  // epilogue staging: per warp one box of 32 rows x 32 columns of bf16 (64-byte
  // rows, 64-byte swizzle: 16-byte chunk q of row r at q ^ ((r >> 1) & 3)),
  // stored to C by a tensor-map bulk store
  static constexpr int kStgCols = 32;
  static constexpr int kStgWarpBytes = 32 * kStgCols * 2;
  static constexpr int kEpiWarps = 8;
  static constexpr int kOffBars = kOffStg + kEpiWarps * kStgWarpBytes;
  static constexpr int kNumBars = 2 * kStages + 2;  // full, empty per stage; acc_full, acc_empty
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // per K block: A scales (2 atoms x 4 columns), then per atom the B scales
  // of both weight row tiles (4 + 4 columns)
  static constexpr int kSfColsPerBlock = 24;
  static constexpr int kSfColsPerStage = kSuperK * kSfColsPerBlock;
  static constexpr int kTmemCols = 512;
  static_assert(BN + kStages * kSfColsPerStage <= kTmemCols, "tensor memory");
  static constexpr int kWarpSf0 = 8, kWarpCopyA = 12, kWarpMma = 13, kWarpCopyB = 14;
  // barrier arrival counts.  full[s]: the CTA's A and B copies and its four
  // scale warps, in the even CTA also the odd CTA's relay; acc_empty (used in
  // the even CTA): the epilogue warps of both CTAs
  static constexpr int kFullArrivalsOdd = 2 + 4;
  static constexpr int kFullArrivals = kFullArrivalsOdd + 1;
  static constexpr int kAccEmptyArrivals = 2 * kEpiWarps;
};

__global__ void __launch_bounds__(PairCfg::kThreads, 1)
    gemm_pair_kernel(const GemmArgs args, int64_t tiles_m, int64_t tiles_n, const __grid_constant__ CUtensorMap c_map) {
  // tiles_m: 256-row pair tiles of C; tiles_n: 256-column tiles of C; tile t
  // is row tile t / tiles_n, column tile t % tiles_n
  using P = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P::kOffBars);  // bytes landed, scales written (even: both CTAs')
  uint64_t* empty = full + P::kStages;                                   // MMAs done with the stage
  uint64_t* acc_full = empty + P::kStages;                               // accumulator complete
  uint64_t* acc_empty = acc_full + 1;                                    // read out (even: by both CTAs)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::kOffMisc + 4);

  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const int64_t pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t KT = args.kt_count;
  const int64_t total = tiles_m * tiles_n;
  const int nss = (int)ceil_div(KT, P::kSuperK);  // stages per tile
  const int64_t a_row_tiles = ceil_div(args.m, kTileRows);
  const int64_t b_row_tiles = ceil_div(args.b_rows, kTileRows);
  auto stage_kblocks = [&](int ss) -> int {
    const int64_t left = KT - (int64_t)ss * P::kSuperK;
    return left < P::kSuperK ? (int)left : P::kSuperK;
  };
  // a barrier of the even CTA, addressed from either CTA of the pair
  auto even_bar = [&](uint64_t* bar) -> uint32_t { return map_cluster(smem_addr(bar), 0); };

  if (threadIdx.x == P::kWarpCopyA * 32) {
    for (int s = 0; s < P::kStages; ++s) {
      mbar_init(&full[s], rank == 0 ? P::kFullArrivals : P::kFullArrivalsOdd);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, P::kAccEmptyArrivals);  // used in the even CTA
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == P::kWarpMma) {
    tmem_alloc_pair(tmem_slot, P::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == P::kWarpCopyA || warp == P::kWarpCopyB) {
    // ------------------------------------------------ bulk-copy producers
    const bool act = warp == P::kWarpCopyA;
    if (lane == 0) {
      // The activation image is written by the preceding kernel: its stream
      // waits for that kernel; the weight stream starts at once.
      if (act) pdl_wait();
      const uint8_t* img = act ? args.a_img : args.b_img;
      uint8_t* ring = smem + (act ? P::kOffA : P::kOffB);
      int64_t g = 0;    // stages issued so far
      int s = 0;        // slot of stage g
      uint32_t ph = 0;  // phase parity of that slot's round
      bool stop = false;
      for (int64_t tile = pair; tile < total && !stop; tile += pairs) {
        const int64_t rt = (act ? tile / tiles_n : tile % tiles_n) * 2 + rank;
        const bool present = rt < (act ? a_row_tiles : b_row_tiles);  // ragged last tile: nothing to copy
        for (int ss = 0; ss < nss; ++ss, ++g) {
          if (!wait_bounded(&empty[s], ph ^ 1, abort_flag)) {
            stop = true;
            break;
          }
          if (present) {
            const uint32_t bytes = (uint32_t)stage_kblocks(ss) * kTileBytes;
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_load(ring + s * P::kStageOpBytes, img + image_block(rt, (int64_t)ss * P::kSuperK, KT), bytes, &full[s]);
          } else {
            mbar_arrive(&full[s]);
          }
          if (++s == P::kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (act && !stop) {
        // The MMA thread's commits arrive on empty[] in both CTAs; the last
        // ones must have landed before this CTA may exit.
        for (int64_t q = g > P::kStages ? g - P::kStages : 0; q < g; ++q)
          wait_bounded(&empty[q % P::kStages], (uint32_t)((q / P::kStages) & 1), abort_flag, kDrainLimitCycles);
      }
      if (*abort_flag) {  // let copies already in flight land before the CTA exits
        for (int64_t q = g > P::kStages ? g - P::kStages : 0; q < g; ++q)
          drain_wait(&full[q % P::kStages], (uint32_t)((q / P::kStages) & 1));
      }
    }
    __syncwarp();
  } else if (warp >= P::kWarpSf0 && warp < P::kWarpSf0 + 4) {
    // ------------------------------------- scale factors into tensor memory
    // Lane l of every 32-lane quadrant holds the 16 bytes of atom row l of an
    // operand block in 4 columns (row groups l, l+32, l+64, l+96; K blocks
    // 0-3), the content tcgen05.cp.32x128b.warpx4 would produce.  Per K
    // block: the A atoms (columns 0-7), then for each atom the two weight row
    // tiles' atoms side by side (8-15, 16-23), which is the 256-row B-scale
    // layout of the pair MMA.  Warp 8 + q writes quadrant q.  The atoms come
    // straight from the operand images: the next stage's loads are in flight
    // while the warp waits for the slot to free.
    const int quad = warp - P::kWarpSf0;
    pdl_wait();  // the activation image is written by the preceding kernel
    uint4 sfv[P::kSuperK][3][2];  // [K block][A, B0, B1][atom]
    auto load_stage = [&](int64_t tile, int ss) {
#pragma unroll
      for (int j = 0; j < P::kSuperK; ++j) {
        const int64_t kt = (int64_t)ss * P::kSuperK + j;
        if (kt >= KT) break;
        const uint8_t* src[3];
        const int64_t art = (tile / tiles_n) * 2 + rank;
        src[0] = art < a_row_tiles ? args.a_img + image_block(art, kt, KT) + kTileDataBytes : nullptr;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int64_t brt = (tile % tiles_n) * 2 + t;
          src[1 + t] = brt < b_row_tiles ? args.b_img + image_block(brt, kt, KT) + kTileDataBytes : nullptr;
        }
        // a missing row tile (ragged edge) gets zero scales; its rows are never stored
#pragma unroll
        for (int o = 0; o < 3; ++o) {
          sfv[j][o][0] = src[o] ? ldg_nc_v4(src[o] + lane * 16) : make_uint4(0, 0, 0, 0);
          sfv[j][o][1] = src[o] ? ldg_nc_v4(src[o] + kAtomBytes + lane * 16) : make_uint4(0, 0, 0, 0);
        }
      }
    };
    int64_t tile = pair;
    int ss = 0, s = 0;
    uint32_t ph = 0;
    if (tile < total) load_stage(tile, 0);
    while (tile < total) {
      // tensor-memory slot s is free once the MMAs of its previous stage completed
      if (!__all_sync(0xFFFFFFFFu, wait_bounded(&empty[s], ph ^ 1, abort_flag))) break;
      tc_fence_after();
      const int cnt = stage_kblocks(ss);
#pragma unroll
      for (int j = 0; j < P::kSuperK; ++j) {
        if (j >= cnt) break;
        const uint32_t col = tmem + ((uint32_t)(quad * 32) << 16) + P::BN + s * P::kSfColsPerStage + j * P::kSfColsPerBlock;
        const uint4 a0 = sfv[j][0][0], a1 = sfv[j][0][1];
        const uint4 b00 = sfv[j][1][0], b01 = sfv[j][1][1], b10 = sfv[j][2][0], b11 = sfv[j][2][1];
        const uint32_t va[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t vb0[8] = {b00.x, b00.y, b00.z, b00.w, b10.x, b10.y, b10.z, b10.w};
        const uint32_t vb1[8] = {b01.x, b01.y, b01.z, b01.w, b11.x, b11.y, b11.z, b11.w};
        tmem_store_8(col, va);
        tmem_store_8(col + 8, vb0);
        tmem_store_8(col + 16, vb1);
      }
      tmem_store_wait();  // the source registers are reused below
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);  // scales in place (the copies arrive with their bytes)
      if (++s == P::kStages) {
        s = 0;
        ph ^= 1;
      }
      if (++ss == nss) {
        ss = 0;
        tile += pairs;
      }
      if (tile < total) load_stage(tile, ss);  // the next stage's atoms, in flight during the next wait
    }
  } else if (warp == P::kWarpMma) {
    if (rank == 1) {
      // ---------------------------------------------------- relay (odd CTA)
      // forwards "this CTA's operand bytes and scales of stage g are in
      // place" to the even CTA, whose MMAs read them (the test hook forwards
      // nothing)
      if (lane == 0 && !args.drop_copies) {
        int s = 0;
        uint32_t ph = 0;
        bool stop = false;
        for (int64_t tile = pair; tile < total && !stop; tile += pairs) {
          for (int ss = 0; ss < nss; ++ss) {
            if (!wait_bounded_poll(&full[s], ph, abort_flag)) {
              stop = true;
              break;
            }
            // Relaxed: the bytes and scales are in place once both phases
            // completed, and a cluster-scope release arrive was measured to
            // stall this thread 0.5-1.2 us on GB300 while the epilogue's
            // stores are in flight.
            mbar_arrive_remote_relaxed(even_bar(&full[s]));
            if (++s == P::kStages) {
              s = 0;
              ph ^= 1;
            }
          }
        }
      }
    } else if (lane == 0) {
      // ------------------------------------------------ MMA issuer (even CTA)
      // The MMA queue is shallow: whatever this thread does between two
      // stages' MMAs shows as idle tensor pipe, so the per-stage work is a
      // few integer adds: descriptors are a base plus the block's offset in
      // 16-byte units (shared addresses stay below 2^18, inside the
      // descriptor's 14-bit field), slot and phase are small counters,
      // never a 64-bit division.
      const uint32_t ie = idesc_mxf4(256, 256, 0, 0), io = idesc_mxf4(256, 256, 2, 2);
      const uint64_t adesc0 = smem_desc(smem_addr(smem + P::kOffA), 0, 1024, kLayoutSwizzle128);
      const uint64_t bdesc0 = smem_desc(smem_addr(smem + P::kOffB), 0, 1024, kLayoutSwizzle128);
      const int64_t kt_whole = args.k / kTileK;  // K blocks with all four 64-K steps
      int s = 0;
      uint32_t ph = 0, it = 0;
      bool aborted = false;
      for (int64_t tile = pair; tile < total && !aborted; tile += pairs, ++it) {
        if (!wait_bounded_poll(acc_empty, (it & 1) ^ 1, abort_flag)) break;  // previous tile read out
        for (int ss = 0; ss < nss; ++ss) {
          if (!wait_bounded_poll(&full[s], ph, abort_flag)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const int cnt = stage_kblocks(ss);
          const uint64_t off0 = (uint64_t)((s * P::kStageOpBytes) >> 4);
          const uint32_t sf0 = tmem + P::BN + s * P::kSfColsPerStage;
          if (cnt == 2 && (int64_t)ss * P::kSuperK + 1 < kt_whole) {  // the usual stage: all eight MMAs in one go
            constexpr uint64_t kNext = kTileBytes >> 4;
            mma_mxf4_pair_kblock2(tmem, adesc0 + off0, bdesc0 + off0, adesc0 + off0 + kNext, bdesc0 + off0 + kNext, ie,
                                  io, sf0, sf0 + 8, sf0 + P::kSfColsPerBlock, sf0 + P::kSfColsPerBlock + 8,
                                  ss > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int j = 0; j < P::kSuperK; ++j) {
              if (j >= cnt) break;
              const uint32_t sf = tmem + P::BN + s * P::kSfColsPerStage + j * P::kSfColsPerBlock;
              const uint32_t acc = (ss > 0 || j > 0) ? 1u : 0u;
              const int64_t kt = (int64_t)ss * P::kSuperK + j;
              const uint64_t off = (uint64_t)((s * P::kStageOpBytes + j * kTileBytes) >> 4);
              const uint64_t ad = adesc0 + off, bd = bdesc0 + off;
              if (kt < kt_whole) {  // a whole K block: its four MMAs in one go
                mma_mxf4_pair_kblock(tmem, ad, bd, ie, io, sf, sf + 8, acc);
              } else {
                const int steps = k_steps(args.k, kt);
                for (int kk = 0; kk < steps; ++kk) {
                  // advancing the start address by 32 bytes = 2 in the descriptor's 16-byte units
                  const uint64_t adv = (uint64_t)(kk * 2);
                  mma_mxf4_pair(tmem, ad + adv, bd + adv, (kk & 1) ? io : ie,
                                sf + (uint32_t)(kk >> 1) * 4, sf + 8 + (uint32_t)(kk >> 1) * 8, (acc || kk > 0) ? 1u : 0u);
                }
              }
            }
          }
          mma_commit_pair(&empty[s], 0x3);
          if (++s == P::kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        mma_commit_pair(acc_full, 0x3);  // fires when this tile's MMAs have completed
      }
    }
    __syncwarp();
  } else if (warp < P::kEpiWarps) {
    // --------------------------------------------- epilogue (warps 0-7)
    // This CTA's 128 accumulator rows: warp w reads the 32 x 128 slice of
    // quadrant w % 4 and column half w / 4 into registers as packed bf16 (64
    // registers) and hands the accumulator back before storing, so the next
    // tile's MMAs wait only for the tensor-memory reads, not for the global
    // stores.
    constexpr int kCols = P::BN / 2;
    const int quad = warp % 4, half = warp / 4;
    uint8_t* box = smem + P::kOffStg + warp * P::kStgWarpBytes;
    const int64_t n_tma = args.n & ~int64_t(7);  // the columns the box stores cover
    uint32_t it = 0;
    for (int64_t tile = pair; tile < total; tile += pairs, ++it) {
      const bool ok = wait_bounded_poll(acc_full, it & 1, abort_flag);
      tc_fence_after();
      uint32_t packed[kCols / 16][8];
#pragma unroll
      for (int c = 0; c < kCols / 16; c += 2) {  // two loads in flight per wait
        uint32_t r[2][16];
        tmem_load_16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * kCols + c * 16), r[0]);
        tmem_load_16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * kCols + c * 16 + 16), r[1]);
        tmem_load_wait();
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            packed[c + u][j] = bf16x2_bits(__uint_as_float(r[u][2 * j]), __uint_as_float(r[u][2 * j + 1]));
      }
      tc_fence_before();
      __syncwarp();
      // Accumulator rows read out: free for the next tile.  The odd CTA's
      // warps arrive on the even CTA's barrier directly; their reads have
      // completed (tcgen05.wait::ld) and nothing is published, so the arrival
      // is relaxed and does not wait for the warp's stores of the previous tile.
      if (lane == 0) {
        if (rank == 0) mbar_arrive(acc_empty);
        else mbar_arrive_remote_relaxed(even_bar(acc_empty));
      }
      if (!ok) continue;
      const int64_t m0 = (tile / tiles_n) * (2 * kTileRows) + rank * kTileRows + quad * 32;
      const int64_t n0 = (tile % tiles_n) * P::BN + half * kCols;
      // 32-column chunks: each lane writes its row's 64 bytes into the warp's
      // swizzled box, then one lane stores the box with a tensor-map bulk
      // store (rows >= m and columns past the map's end are not written)
#pragma unroll
      for (int cc = 0; cc < kCols / P::kStgCols; ++cc) {
        if (lane == 0) bulk_wait_group_read0();  // the previous store has read the box
        __syncwarp();
        uint8_t* row_dst = box + lane * (P::kStgCols * 2);
#pragma unroll
        for (int q = 0; q < P::kStgCols / 8; ++q) {
          const int c = cc * (P::kStgCols / 16) + (q >> 1), h = q & 1;
          *reinterpret_cast<uint4*>(row_dst + ((q ^ ((lane >> 1) & 3)) << 4)) =
              make_uint4(packed[c][4 * h], packed[c][4 * h + 1], packed[c][4 * h + 2], packed[c][4 * h + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int64_t x0 = n0 + cc * P::kStgCols;
        if (lane == 0) {
          tma_store_2d(&c_map, box, (int)x0, (int)m0);
          bulk_commit_group();
        }
        // The tensor map ends at n rounded down to 8 columns (the copy engine
        // clips whole 16-byte chunks only); the last n mod 8 columns of a row
        // are stored here, from the same box.
        if (x0 + P::kStgCols > n_tma && x0 < args.n && m0 + lane < args.m) {
          for (int64_t col = n_tma > x0 ? n_tma : x0; col < args.n && col < x0 + P::kStgCols; ++col) {
            const int j = (int)(col - x0);
            const uint16_t v = *reinterpret_cast<const uint16_t*>(
                row_dst + ((((j * 2) >> 4) ^ ((lane >> 1) & 3)) << 4) + ((j * 2) & 15));
            *reinterpret_cast<uint16_t*>(args.c + (m0 + lane) * args.ldc + col) = v;
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store of this warp has completed
  }

  // Neither CTA frees its tensor memory or exits while the pair still needs
  // it: every MMA has completed (both epilogues waited for the last
  // accumulator), every remote arrival has been made.
  tc_fence_before();
  cluster_sync();
  if (warp == P::kWarpMma) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P::kTmemCols);
  }
}

// ------------------------------------------------------------------ host
// The host-side caches below are per device and idempotent (two threads that
// miss at once compute or set the same value), so relaxed atomics suffice to
// keep concurrent callers race-free.
int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (v <= 0) v = 148;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Testing and tuning overrides: the K-split factor the planner picks
// (0 = its own choice, else 1 to 8, clamped to what the shape and the
// kernel allow) and the copy-dropping hook of the failure-detection test.
// Read from MXFP4_SPLIT_K and MXFP4_DEBUG_DROP_COPIES once, when the library
// is loaded, and changed afterwards only through set_debug_options: no call
// of the GEMM reads the environment.
static int env_split() {
  const char* v = getenv("MXFP4_SPLIT_K");
  const int s = v ? atoi(v) : 0;
  return (s >= 1 && s <= 8) ? s : 0;
}
static int env_drop() {
  const char* v = getenv("MXFP4_DEBUG_DROP_COPIES");
  return (v && v[0] == '1') ? 1 : 0;
}
static std::atomic<int> g_split_override{env_split()};
static std::atomic<int> g_drop_copies{env_drop()};

static int split_override() { return g_split_override.load(std::memory_order_relaxed); }

bool set_debug_options(int split_k, int drop_copies) {
  if (split_k < 0 || split_k > 8) return false;
  if (drop_copies != 0 && drop_copies != 1) return false;
  g_split_override.store(split_k, std::memory_order_relaxed);
  g_drop_copies.store(drop_copies, std::memory_order_relaxed);
  return true;
}

int kernel_binary_version() {
  cudaFuncAttributes attr{};
  if (cudaFuncGetAttributes(&attr, gemm_kernel<32, kFusedSwap>) != cudaSuccess) return -1;
  return attr.binaryVersion;
}

int make_gemm_plan(int64_t m, int64_t n, int64_t k, GemmPlan* plan, bool a_image) {
  const int sms = num_sms();
  const int forced = split_override();
  const int64_t KT = ceil_div(k, kTileK);
  GemmPlan p{};
  if (m <= 128) {
    p.swap_ab = true;
    p.mode = (m <= 32 && !a_image) ? kFusedSwap : kImageSwap;
    p.bn = p.mode == kFusedSwap ? (m <= 16 ? 16 : 32) : (m <= 64 ? 64 : 128);
    p.grid_x = ceil_div(n, kTileRows);
    const int s_max = 8;  // the kernels' kMaxSplit
    // The cluster exchange of a split costs about 1-1.5 us (measured on
    // GB300 for m <= 64); a 256-K block of weights streams in a fraction of
    // that, so a split pays only while every rank keeps several K blocks.
    // The fused kernel (m <= 32) streams only weights, and the rate at which
    // one SM receives them is what bounds it after an L2 flush, so it takes
    // the most ranks that fit on the SMs with at least 4 K blocks each
    // (k = 7168 with n = 2112: 6 ranks, 102 CTAs); the image kernels keep
    // power-of-two splits with at least 5 K blocks per rank (k = 512 and
    // 2048 run unsplit).
    int s = 1;
    if (p.mode == kFusedSwap) {
      while (s < s_max && p.grid_x * (s + 1) <= sms && KT >= 4 * (s + 1)) ++s;
    } else {
      while (s < s_max && p.grid_x * s * 2 <= sms && KT / (s * 2) >= 5) s *= 2;
    }
    if (forced) s = forced <= KT ? forced : 1;
    p.split = s;
    p.grid_y = s;
    p.workspace = (p.mode == kFusedSwap || a_image) ? 0 : (size_t)image_bytes(m, k);
  } else {
    p.swap_ab = false;
    p.mode = kImagePlain;
    const int64_t mt = ceil_div(m, kTileRows);
    // the CTA-pair kernel wants at least one full 256-column tile (its C box
    // stores need n >= 8) and a tile per SM
    p.bn = (n >= 256 && mt * ceil_div(n, 256) >= sms) ? 256 : 128;
    p.grid_x = mt;
    const int64_t nt = ceil_div(n, p.bn);
    const int s_max = p.bn == 256 ? 1 : 8;  // the kernels' kMaxSplit
    int s = 1;
    while (s < s_max && mt * nt * s * 2 <= sms && KT / (s * 2) >= 4) s *= 2;
    if (forced) s = (forced <= KT && forced <= s_max) ? forced : 1;
    p.split = s;
    p.grid_y = nt * s;
    p.workspace = a_image ? 0 : (size_t)image_bytes(m, k);
    if (p.bn == 256) {  // at least one 128 x 256 tile per SM: CTA pairs loop over 256 x 256 tiles
      p.persistent = true;
      const int64_t pair_tiles = ceil_div(m, 2 * kTileRows) * nt;
      p.grid_x = 2 * (pair_tiles < sms / 2 ? pair_tiles : sms / 2);
      p.grid_y = 1;
    }
  }
  if (p.grid_x > 0x7FFFFFFF || p.grid_y > 65535) return 1;
  *plan = p;
  return 0;
}

// Thread-block clusters of a given size that can be resident at once for this
// kernel (cached per device and cluster size).
template <int BN, int kMode>
static int max_resident_clusters(int split) {
  using C = Cfg<BN, kMode>;
  static std::atomic<int> cache[64][9];  // [device][split]
  int dev = 0;
  cudaGetDevice(&dev);
  const int idx = split >= 0 && split <= 8 ? split : 0;
  if (dev < 0 || dev >= 64) return 0;
  const int hit = cache[dev][idx].load(std::memory_order_relaxed);
  if (hit != 0) return hit;
  {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, (unsigned)split, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = (unsigned)split;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<BN, kMode>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();  // clear the error: the launch decides
      n = -1;
    }
    cache[dev][idx].store(n, std::memory_order_relaxed);
    return n;
  }
}

template <int BN, int kMode>
static cudaError_t launch_one(const GemmPlan& plan_in, const GemmArgs& args_in, cudaStream_t stream) {
  using C = Cfg<BN, kMode>;
  if (plan_in.split > C::kMaxSplit) return cudaErrorInvalidConfiguration;
  static std::atomic<bool> attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  // A K split whose clusters cannot all be resident at once would run in two
  // waves; reduce it until they fit (the result does not depend on the split
  // beyond the fp32 summation order).
  GemmPlan plan = plan_in;
  GemmArgs args = args_in;
  while (plan.split > 1) {
    const int fit = max_resident_clusters<BN, kMode>(plan.split);
    if (fit < 0 || (int64_t)fit * plan.split >= plan.grid_x * plan.grid_y) break;
    plan.grid_y = plan.grid_y / plan.split * (plan.split - 1);
    plan.split -= 1;
  }
  args.split = plan.split;
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

// CTA pairs of the pair kernel that can be resident at once (cached per device).
static int max_resident_pairs() {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 0;
  const int hit = cache[dev].load(std::memory_order_relaxed);
  if (hit != 0) return hit;
  {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(PairCfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();  // clear the error: the launch decides
      n = -1;
    }
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
  }
}

// The tensor map of C (bf16 [m, n], row stride ldc) for the pair kernel's
// box stores: boxes of 32 rows x 32 columns, 64-byte swizzle.  The encoder
// comes from the driver through the runtime's entry-point query.
static cudaError_t encode_c_map(const GemmArgs& args, CUtensorMap* map) {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 encode = cached.load(std::memory_order_relaxed);
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cached.store(encode, std::memory_order_relaxed);
  }
  // n rounded down to 8 columns: the copy engine clips whole 16-byte chunks,
  // so a map to n itself would write up to 7 columns past it
  const cuuint64_t dims[2] = {(cuuint64_t)(args.n & ~int64_t(7)), (cuuint64_t)args.m};
  const cuuint64_t strides[1] = {(cuuint64_t)args.ldc * 2};
  const cuuint32_t box[2] = {(cuuint32_t)PairCfg::kStgCols, 32};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, args.c, dims, strides, box, elem_strides,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static cudaError_t launch_pair(const GemmPlan& plan, const GemmArgs& args, int64_t tiles_m, int64_t tiles_n,
                               cudaStream_t stream) {
  static std::atomic<bool> attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  int64_t pairs = plan.grid_x / 2;
  const int resident = max_resident_pairs();
  if (resident > 0 && pairs > resident) pairs = resident;  // one wave: every pair loops over its tiles
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(PairCfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // dependent of the quantization kernel
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  // The map depends only on C's address and shape: each host thread keeps
  // its last few, so repeated calls on the same output skip the encoding.
  struct MapEntry {
    const void* c;
    int64_t m, n, ldc;
    CUtensorMap map;
  };
  thread_local MapEntry recent[4] = {};
  thread_local int next_slot = 0;
  const CUtensorMap* c_map = nullptr;
  for (const MapEntry& r : recent)
    if (r.c == args.c && r.m == args.m && r.n == args.n && r.ldc == args.ldc) c_map = &r.map;
  if (!c_map) {
    MapEntry& r = recent[next_slot];
    next_slot = (next_slot + 1) & 3;
    r.c = nullptr;
    const cudaError_t e = encode_c_map(args, &r.map);
    if (e != cudaSuccess) return e;
    r.c = args.c;
    r.m = args.m;
    r.n = args.n;
    r.ldc = args.ldc;
    c_map = &r.map;
  }
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel, args, tiles_m, tiles_n, *c_map);
}

cudaError_t launch_gemm(const GemmPlan& plan, const void* a_bf16, int64_t m, int64_t k, int64_t lda,
                        const void* b_image, int64_t n, void* c, int64_t ldc, void* workspace,
                        cudaStream_t stream, const void* a_image) {
  GemmArgs args{};
  args.m = m;
  args.n = n;
  args.k = k;
  args.kt_count = ceil_div(k, kTileK);
  args.c = static_cast<__nv_bfloat16*>(c);
  args.ldc = ldc;
  args.split = plan.split;
  args.lda = lda;
  // The copy-dropping hook exercises the bounded waits from the tests: the
  // generic GEMM issues no bulk copies, the CTA-pair GEMM's relay forwards
  // nothing; either way the MMA issuer's wait runs out after about a second,
  // the kernel sets the device timeout flag, winds down and exits normally.
  args.drop_copies = g_drop_copies.load(std::memory_order_relaxed);
  if (plan.mode == kFusedSwap) {
    args.a_img = static_cast<const uint8_t*>(b_image);
    args.act = static_cast<const uint16_t*>(a_bf16);
    switch (plan.bn) {
      case 16: return launch_one<16, kFusedSwap>(plan, args, stream);
      case 32: return launch_one<32, kFusedSwap>(plan, args, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (!a_image) {
    cudaError_t e = launch_quant_image(a_bf16, m, k, lda, workspace, stream);
    if (e != cudaSuccess) return e;
    a_image = workspace;
  }
  if (plan.mode == kImageSwap) {
    args.a_img = static_cast<const uint8_t*>(b_image);
    args.b_img = static_cast<const uint8_t*>(a_image);
    args.b_rows = m;
    switch (plan.bn) {
      case 64: return launch_one<64, kImageSwap>(plan, args, stream);
      case 128: return launch_one<128, kImageSwap>(plan, args, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  args.a_img = static_cast<const uint8_t*>(a_image);
  args.b_img = static_cast<const uint8_t*>(b_image);
  args.b_rows = n;
  if (plan.persistent) return launch_pair(plan, args, ceil_div(m, 2 * kTileRows), ceil_div(n, PairCfg::BN), stream);
  switch (plan.bn) {
    case 128: return launch_one<128, kImagePlain>(plan, args, stream);
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
