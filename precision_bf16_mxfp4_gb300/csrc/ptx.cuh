// Inline-PTX wrappers for the sm_103a features the MXFP4 kernels use:
// mbarriers, bulk (TMA-engine) copies, tcgen05 tensor-memory allocation,
// block-scaled MMA, scale-factor copies and accumulator loads, cluster
// shared-memory access and programmatic dependent launch.
#pragma once
#include <cstdint>

namespace mxfp4 {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------ async proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Barrier among `threads` threads (whole warps) of the CTA on hardware
// barrier `id` (0 is the one __syncthreads uses).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bulk copy global -> shared through the TMA engine; completion is counted
// in bytes on `bar`.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Same, with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void bulk_load_hint(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem, fp32) (+)= A(smem, e2m1) * B(smem, e2m1)^T with per-32-element
// e8m0 scale factors for A and B read from tensor memory; K = 64 per call.
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// The four MMAs of one 256-K block (four 64-K steps) into one accumulator,
// from one asm block with every operand ready (see below).
__device__ __forceinline__ void mma_mxf4_kblock(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc_even,
                                                uint32_t idesc_odd, uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, c1, c2, c3;\n\t.reg .b32 sa1, sb1;\n\t"
      "setp.ne.b32 p, %7, 0;\n\tsetp.eq.b32 q, %7, %7;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 c1, %2, 2;\n\tadd.s64 c2, %2, 4;\n\tadd.s64 c3, %2, 6;\n\t"
      "add.u32 sa1, %5, 4;\n\tadd.u32 sb1, %6, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a1, c1, %4, [%5], [%6], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a2, c2, %3, [sa1], [sb1], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a3, c3, %4, [sa1], [sb1], q;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc_even), "r"(idesc_odd), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// The eight MMAs of one 256-K block for a 128 x 256 accumulator held as two
// N = 128 halves (d, d + 128): four 64-K steps, each into both halves.  One
// asm block with every operand ready: the MMA queue is shallow, so address
// arithmetic between single MMAs would leave the tensor pipe idle.  The
// descriptors advance 32 bytes (2 units) per step; scale ids alternate 0/2
// (even/odd idesc); the scale columns advance 4 per two steps.
__device__ __forceinline__ void mma_mxf4_kblock_n256(uint32_t d, uint64_t a, uint64_t b0, uint64_t b1,
                                                     uint32_t idesc_even, uint32_t idesc_odd, uint32_t sfa,
                                                     uint32_t sfb0, uint32_t sfb1, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, c1, c2, c3, e1, e2, e3;\n\t.reg .b32 d1, sa1, sb1, sc1;\n\t"
      "setp.ne.b32 p, %9, 0;\n\tsetp.eq.b32 q, %9, %9;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 c1, %2, 2;\n\tadd.s64 c2, %2, 4;\n\tadd.s64 c3, %2, 6;\n\t"
      "add.s64 e1, %3, 2;\n\tadd.s64 e2, %3, 4;\n\tadd.s64 e3, %3, 6;\n\t"
      "add.u32 d1, %0, 128;\n\tadd.u32 sa1, %6, 4;\n\tadd.u32 sb1, %7, 4;\n\tadd.u32 sc1, %8, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %4, [%6], [%7], p;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [d1], %1, %3, %4, [%6], [%8], p;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a1, c1, %5, [%6], [%7], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [d1], a1, e1, %5, [%6], [%8], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a2, c2, %4, [sa1], [sb1], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [d1], a2, e2, %4, [sa1], [sc1], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a3, c3, %5, [sa1], [sb1], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [d1], a3, e3, %5, [sa1], [sc1], q;\n\t}"
      ::"r"(d), "l"(a), "l"(b0), "l"(b1), "r"(idesc_even), "r"(idesc_odd), "r"(sfa), "r"(sfb0), "r"(sfb1),
      "r"(accumulate)
      : "memory");
}

// ---------------------------------------------- CTA-pair (cta_group::2) forms
// Tensor memory of a CTA pair is allocated, released and freed collectively:
// one warp of each of the two CTAs executes the instruction, and both CTAs
// receive the same base address (measured on GB300).  A kernel uses either
// these forms or the cta_group::1 ones, never both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// One K = 64 step of a 256 x N pair MMA, issued by one thread of the even
// CTA: rows 0-127 of A and D live in the even CTA (its shared memory and
// tensor memory), rows 128-255 in the odd one, at the same addresses; B's
// first N/2 rows come from the even CTA's shared memory, the rest from the
// odd CTA's.  Scales: each CTA's tensor memory holds the A scales of its own
// 128 rows (row r at lane r, column r/32) and the B scales of all N rows
// (row j at column j/32, lane j mod 32 of every 32-lane quadrant) - the
// placement measured on GB300.
__device__ __forceinline__ void mma_mxf4_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                              uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// The four K = 64 steps of one 256-K block of a 256 x 256 pair MMA, from one
// asm block.  A scales advance 4 columns per two steps (128 rows per atom),
// B scales 8 (256 rows).
__device__ __forceinline__ void mma_mxf4_pair_kblock(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc_even,
                                                     uint32_t idesc_odd, uint32_t sfa, uint32_t sfb,
                                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, c1, c2, c3;\n\t.reg .b32 sa1, sb1;\n\t"
      "setp.ne.b32 p, %7, 0;\n\tsetp.eq.b32 q, %7, %7;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 c1, %2, 2;\n\tadd.s64 c2, %2, 4;\n\tadd.s64 c3, %2, 6;\n\t"
      "add.u32 sa1, %5, 4;\n\tadd.u32 sb1, %6, 8;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], a1, c1, %4, [%5], [%6], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], a2, c2, %3, [sa1], [sb1], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], a3, c3, %4, [sa1], [sb1], q;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc_even), "r"(idesc_odd), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Two consecutive 256-K blocks of a 256 x 256 pair MMA (eight MMAs) from
// one asm block: the second block's operands at a2 / b2 and its scales at
// sfa2 / sfb2 (same layout as the first's).
__device__ __forceinline__ void mma_mxf4_pair_kblock2(uint32_t d, uint64_t a, uint64_t b, uint64_t a2, uint64_t b2,
                                                      uint32_t idesc_even, uint32_t idesc_odd, uint32_t sfa,
                                                      uint32_t sfb, uint32_t sfa2, uint32_t sfb2,
                                                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a3, a5, c1, c3, c5, e1, e3, e5, f1, f3, f5;\n\t"
      ".reg .b32 sa1, sb1, sa3, sb3;\n\t"
      "setp.ne.b32 p, %11, 0;\n\tsetp.eq.b32 q, %11, %11;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a3, %1, 4;\n\tadd.s64 a5, %1, 6;\n\t"
      "add.s64 c1, %2, 2;\n\tadd.s64 c3, %2, 4;\n\tadd.s64 c5, %2, 6;\n\t"
      "add.s64 e1, %3, 2;\n\tadd.s64 e3, %3, 4;\n\tadd.s64 e5, %3, 6;\n\t"
      "add.s64 f1, %4, 2;\n\tadd.s64 f3, %4, 4;\n\tadd.s64 f5, %4, 6;\n\t"
      "add.u32 sa1, %7, 4;\n\tadd.u32 sb1, %8, 8;\n\tadd.u32 sa3, %9, 4;\n\tadd.u32 sb3, %10, 8;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %5, [%7], [%8], p;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], a1, c1, %6, [%7], [%8], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], a3, c3, %5, [sa1], [sb1], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], a5, c5, %6, [sa1], [sb1], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %3, %4, %5, [%9], [%10], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], e1, f1, %6, [%9], [%10], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], e3, f3, %5, [sa3], [sb3], q;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], e5, f5, %6, [sa3], [sb3], q;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "l"(a2), "l"(b2), "r"(idesc_even), "r"(idesc_odd), "r"(sfa), "r"(sfb), "r"(sfa2),
      "r"(sfb2), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in each CTA of `cta_mask`
// when every tcgen05 operation this thread issued before it has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(cta_mask)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_load_16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_load_32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Each thread of the warp writes 8 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_store_8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_store_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_load_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (16-byte units), version 1, layout/swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}
constexpr uint32_t kLayoutSwizzle128 = 2;
constexpr uint32_t kLayoutNoSwizzle = 0;

// Instruction descriptor for kind::mxf4 (E2M1 x E2M1, UE8M0 scales, fp32
// accumulator implied, both operands K-major, dense K = 64).
__host__ __device__ constexpr uint32_t idesc_mxf4(uint32_t m, uint32_t n, uint32_t sfa_id, uint32_t sfb_id) {
  return ((sfb_id & 3u) << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24) |
         ((sfa_id & 3u) << 29);
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (address from
// map_cluster), releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_caddr) : "memory");
}
// The same arrival without release semantics: for hand-offs that publish no
// memory (say, "these tensor-memory reads have completed"), so the thread
// need not wait for its earlier global stores to be performed first.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t bar_caddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_caddr) : "memory");
}
// try_wait that acquires writes released at cluster scope by other CTAs.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase, acquiring at cluster scope.  A thread that
// polls with it sees an arrival from another CTA as soon as it lands; a
// try_wait that suspended the thread was measured on GB300 to resume some
// 0.5-1 us after such an arrival.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint32_t map_cluster(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Bulk copy from this CTA's shared memory into another CTA's shared memory
// in the cluster; the bytes complete on an mbarrier in the destination CTA.
// 16-byte aligned addresses, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_caddr, const void* src_smem, uint32_t bytes,
                                                     uint32_t mbar_caddr) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_caddr),
      "r"(smem_addr(src_smem)), "r"(bytes), "r"(mbar_caddr)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Tiled bulk store of a 2-D box from this CTA's shared memory to global
// memory through a tensor map (a kernel parameter); coordinates (x, y) in
// elements, x innermost.  Elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void* tensor_map, const void* src_smem, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tensor_map)),
               "r"(smem_addr(src_smem)), "r"(x), "r"(y)
               : "memory");
}
// Wait until this thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Wait until the source buffers of this thread's committed bulk copies have been read.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ------------------------------------------------ programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

}  // namespace mxfp4
