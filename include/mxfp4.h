/*
 * mxfp4.h -- C ABI of the GB300 (sm_103a) MXFP4 GEMM library.
 *
 *   C[m,n] = quant(A) . B^T
 *
 * A is bf16 [m,k], quantized on the fly to MXFP4 (e2m1 values with one e8m0
 * scale per 32 consecutive K elements); B is MXFP4 [n,k], quantized ahead of
 * time; C is bf16 [m,n] with fp32 accumulation.
 *
 * The operation is the one benchmarked by the "kernelbot amd-mxfp4-mm"
 * submission pages: the quantizer of submission 694791 ("MXFP4
 * quantization: bf16 -> fp4(e2m1) + e8m0 block scales") and the
 * `tl.dot_scaled(a, a_scale, "e2m1", b, b_scale, "e2m1", acc)` product of
 * submission 752099, whose harness entry takes (A, B, B_q, B_shuffle,
 * B_scale) and returns C.
 *
 * Conventions for every entry point
 *   - Pointers named *_bf16 / a_fp4 / a_scale / b_* / c_* / workspace are
 *     DEVICE pointers of the current CUDA device, except a_host / c_host of
 *     mxfp4_gemm_host; the caller allocates and owns them.  The library
 *     never allocates, never synchronizes (except mxfp4_device_status and
 *     the mxfp4_measure_fp4_peak measurement) and only enqueues work on
 *     `stream`.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - Element strides (lda, ldc) are in elements, row-major.
 *   - Errors: MXFP4_ERR_INVALID_ARG / MXFP4_ERR_UNSUPPORTED are returned
 *     before anything is enqueued; MXFP4_ERR_CUDA reports a launch failure
 *     (the error status of the launch itself); faults that happen later
 *     surface at the caller's next synchronization, as with any CUDA call.
 *   - Entry points may be called from several host threads and on several
 *     streams at once.  The state the library keeps: per device, cached
 *     kernel attributes and occupancy figures, and the watchdog flag of
 *     mxfp4_device_status (a device variable every kernel of the library
 *     may set); per host thread, the last few tensor maps of C the
 *     large-m GEMM was launched with, and per host thread and device the
 *     helper stream and five events of mxfp4_gemm_host's chunked round trip
 *     (created on first use, never destroyed); per process, the overrides of
 *     mxfp4_set_debug_options.  The exception is mxfp4_gemm_noalloc: its
 *     scratch is one device array shared by every call on a device, so
 *     calls of it that overlap on the GPU race (see its declaration).
 *   - Bounded waits and timeouts: every wait inside a GEMM kernel gives up
 *     after about 2^31 SM clock cycles (~1 s at 2 GHz).  The cycle counter
 *     keeps running while the context is switched out, so a GPU time-sliced
 *     with another busy context can reach the limit on a valid call.  A
 *     kernel that gives up sets the watchdog flag and leaves C undefined
 *     (partly written); it reports this only through mxfp4_device_status,
 *     which callers that need to know must call after the GEMM.
 */
#ifndef MXFP4_H_
#define MXFP4_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MXFP4_API __attribute__((visibility("default")))
#else
#define MXFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXFP4_OK = 0,
  MXFP4_ERR_INVALID_ARG = 1, /* null/unaligned pointer, bad size or stride */
  MXFP4_ERR_UNSUPPORTED = 2, /* valid arguments this build does not handle */
  MXFP4_ERR_WORKSPACE = 3,   /* workspace smaller than mxfp4_gemm_workspace_bytes */
  MXFP4_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  MXFP4_ERR_TIMEOUT = 5      /* a kernel's bounded pipeline wait ran out */
} mxfp4_status;

/* Static, NUL-terminated name of a status code. */
MXFP4_API const char* mxfp4_status_string(int status);

/* Library ABI version (major * 100 + minor). */
MXFP4_API int mxfp4_version(void);

/*
 * mxfp4_quant -- bf16 A[m,k] (row stride lda elements) -> MXFP4.
 *   a_fp4   : u8 [m, k/2], dense; byte j of a row = code(2j) | code(2j+1) << 4
 *             (even K index in the low nibble), code = sign bit 3 | e2m1 magnitude.
 *   a_scale : u8 [m, k/32], dense; e8m0 byte = ub + 127.
 * Block rule (submission 694791, "MXFP4 quantization"): per 32 consecutive
 * elements, amax -> fp32 bits + 0x200000, & 0xFF800000 -> exponent field -
 * 129 = ub, clamped to [-127, 127]; each element x is encoded as
 * e2m1(x * 2^-ub), rounded to nearest even, saturating at 6.0; a negative
 * value rounding to zero keeps its sign (nibble 0x8).  Subnormal inputs are
 * exact; NaN/Inf inputs give unspecified codes.
 * Preconditions: m >= 0, k > 0, k % 32 == 0, lda >= k, lda % 8 == 0, all
 * pointers 16-byte aligned (a_scale: any alignment).  m == 0 is a no-op.
 */
MXFP4_API mxfp4_status mxfp4_quant(const void* a_bf16, int64_t m, int64_t k, int64_t lda, void* a_fp4, void* a_scale,
                         void* stream);

/*
 * Size in bytes of the prepacked image of an MXFP4 B[n,k] (0 if n <= 0,
 * k <= 0 or k % 32 != 0).  The pages hand B to the GEMM already
 * quantized and shuffled into their kernel's layout (submission 752099,
 * `custom_kernel` input tuple: B_q and B_shuffle, B_scale); this is the
 * size of the GB300 form of that pre-shuffled weight: ceil(n/128) x
 * ceil(k/256) blocks of 17,408 bytes (16 KiB of e2m1 data, 1 KiB of e8m0
 * scales).
 */
MXFP4_API size_t mxfp4_prepacked_b_bytes(int64_t n, int64_t k);

/*
 * mxfp4_prepack_b -- one-time repack of MXFP4 B into the layout the tensor
 * cores read: tiles of 128 rows x 256 K elements, data in the 128-byte
 * swizzled K-major order and e8m0 scales in the 32-lane x 16-byte atoms
 * of a tensor-memory lane quadrant's scale columns.  This replaces the pages'
 * AMD-specific B_shuffle / `e8m0_shuffle` scale layout (submission 739530,
 * `_sh_row` / `_sh_col`), which exists only for the MI355X MFMA lane order.
 *   b_fp4   : u8 [n, k/2] as produced by mxfp4_quant (dense rows)
 *   b_scale : u8 [n, k/32] as produced by mxfp4_quant (dense rows)
 *   b_packed: u8 [b_packed_bytes], opaque; valid only for this (n, k).
 * Preconditions: n > 0, k > 0, k % 32 == 0, b_packed_bytes >=
 * mxfp4_prepacked_b_bytes(n, k), b_fp4 and b_packed 16-byte aligned.
 */
MXFP4_API mxfp4_status mxfp4_prepack_b(const void* b_fp4, const void* b_scale, int64_t n, int64_t k, void* b_packed,
                             size_t b_packed_bytes, void* stream);

/*
 * Workspace bytes mxfp4_gemm needs for this shape: 0 for m <= 32, where
 * quantized A never leaves shared memory; otherwise the size of A's tiled
 * operand image (the same formula as mxfp4_prepacked_b_bytes(m, k)).  The
 * pages choose by M between quantizing A inside the GEMM and a separate
 * quantization pass whose output the GEMM reads (submission 739530, v10h
 * docstring: the fused path for small M, a prequantized A for larger M;
 * submission 694791, module docstring, "Two kernel paths depending on K");
 * the workspace holds that intermediate for the second path.  0 also for
 * invalid arguments.
 */
MXFP4_API size_t mxfp4_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k);

/*
 * mxfp4_gemm -- C[m,n] (row stride ldc) = bf16( quant(A) . B^T ), fp32
 * accumulation; the summation order is unspecified but deterministic for a
 * given shape and device.  The operation of submission 752099
 * (`_quant_gemm_fused_launcher`: A quantized with the rule of mxfp4_quant,
 * then `tl.dot_scaled(a, a_scale, "e2m1", b, b_scale, "e2m1", acc)` with an
 * fp32 accumulator, stored as `acc.to(bf16)`): every product of two e2m1
 * values and their two power-of-two scales is exact, so C differs from the
 * exact sum only by the fp32 summation order and the final rounding.
 *   a_bf16   : bf16 [m, k], row stride lda elements
 *   b_packed : image from mxfp4_prepack_b for (n, k)
 *   c_bf16   : bf16 [m, n], row stride ldc elements (written, not read)
 *   workspace: device scratch of at least mxfp4_gemm_workspace_bytes(m,n,k)
 *              bytes (may be NULL when that is 0); 16-byte aligned.
 * m <= 32: one launch; A is quantized inside the GEMM kernel.  m > 32: a
 * quantization launch writes A's operand image into the workspace and the
 * GEMM launch reads it; the GEMM is a programmatic dependent launch that
 * streams its first weight tiles while the quantization runs.  When K is
 * split across a thread-block cluster, partial sums are added in a fixed
 * order, so results are bitwise reproducible.
 * Preconditions: m, n > 0, k > 0, k % 32 == 0, lda >= k, lda % 8 == 0,
 * ldc >= n, ldc % 8 == 0, a_bf16 / b_packed / c_bf16 16-byte aligned.
 */
MXFP4_API mxfp4_status mxfp4_gemm(const void* a_bf16, int64_t m, int64_t k, int64_t lda, const void* b_packed, int64_t n,
                        void* c_bf16, int64_t ldc, void* workspace, size_t workspace_bytes, void* stream);

/*
 * mxfp4_gemm_host -- mxfp4_gemm for an A that lives in host memory and a C
 * that is wanted there: on `stream`, one 2-D copy of A to the device, the
 * GEMM of mxfp4_gemm, one 2-D copy of C back.  The pages' entry point takes
 * its input tuple and returns C (submission 752099, `custom_kernel`); this is
 * that round trip for a caller whose tensors are in host memory.  When C is
 * at least 8 MiB (m > 32, m >= 512) the round trip runs in up to four chunks
 * of whole 256-row tiles: each chunk's A copy and GEMM on `stream`, its C
 * copy on a helper stream of the library after that GEMM, so that the
 * downloads overlap the later chunks; `stream` then waits for the last
 * download, so work enqueued on it after the call sees the whole C.  During
 * stream capture the chunked form is used only if the helper stream already
 * exists (an earlier call on this host thread and device created it);
 * otherwise the call takes the single-stream form.
 *   a_host   : bf16 [m, k] in host memory, row stride lda elements
 *   b_packed : image from mxfp4_prepack_b for (n, k), in device memory
 *   c_host   : bf16 [m, n] in host memory, row stride ldc elements (written)
 *   a_dev    : device staging for A, bf16 [m, k] with row stride k
 *   c_dev    : device staging for C, bf16 [m, n8] with n8 = n rounded up to
 *              a multiple of 8 (row stride n8)
 *   workspace: as mxfp4_gemm
 * With page-locked host buffers the call only enqueues; C is complete in
 * c_host once `stream` has passed the call (synchronize before reading it).
 * With page-locked buffers whose row strides are multiples of 8 elements
 * (16-byte aligned rows), the kernels read A from and write C to host memory
 * directly (mapped into the device's address space; over NVLink-C2C on
 * GB300) and the staging buffers are not touched, except for the large-m
 * CTA-pair plan (C stored by tensor-map bulk copies) and for m <= 32 with
 * k > 512 (A read in several rounds of host round trips); those take the two
 * copies through a_dev and c_dev.  With pageable host buffers the
 * runtime stages the copies and the call may block.  The caller owns every
 * buffer; nothing is allocated.
 * Preconditions: m, n > 0, k > 0, k % 32 == 0, lda >= k, ldc >= n, host
 * pointers non-null, a_dev / c_dev / b_packed 16-byte aligned.
 * Errors: MXFP4_ERR_INVALID_ARG, MXFP4_ERR_WORKSPACE, MXFP4_ERR_UNSUPPORTED,
 * MXFP4_ERR_CUDA (a copy or a launch failed to enqueue).
 */
MXFP4_API mxfp4_status mxfp4_gemm_host(const void* a_host, int64_t m, int64_t k, int64_t lda, const void* b_packed,
                                       int64_t n, void* c_host, int64_t ldc, void* a_dev, void* c_dev,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * mxfp4_prepack_b_bf16 -- the on-device weight path in one call: bf16 B[n,k]
 * (row stride ldb) straight into the prepacked image, bit-identical to
 * mxfp4_quant followed by mxfp4_prepack_b, with no intermediate buffer.  The
 * pages hand B in bf16 beside its MXFP4 form (submission 752099,
 * `custom_kernel` input tuple); this quantizes it with the same rule as A.
 *   b_bf16  : bf16 [n, k], row stride ldb elements
 *   b_packed: u8 [b_packed_bytes], opaque; valid only for this (n, k).
 * Preconditions: n > 0, k > 0, k % 32 == 0, ldb >= k, ldb % 8 == 0,
 * b_packed_bytes >= mxfp4_prepacked_b_bytes(n, k), b_bf16 and b_packed
 * 16-byte aligned.  Errors: MXFP4_ERR_INVALID_ARG, MXFP4_ERR_CUDA.
 */
MXFP4_API mxfp4_status mxfp4_prepack_b_bf16(const void* b_bf16, int64_t n, int64_t k, int64_t ldb, void* b_packed,
                                            size_t b_packed_bytes, void* stream);

/*
 * Reusing one quantized activation across several GEMMs (the pages' fused
 * "quant + scale-shuffle write" of the activation, submission 705642 v3
 * docstring, lifted into its own call): mxfp4_quant_image writes A's MXFP4
 * quantization directly in the tensor-core operand layout (scales already in
 * the tensor-memory atom order), and mxfp4_gemm_image multiplies such an
 * image by any prepacked B of the same k without quantizing again.
 *
 * mxfp4_act_image_bytes(m, k): bytes of the activation image (the same
 * formula as mxfp4_prepacked_b_bytes(m, k)); 0 for invalid arguments.
 *
 * mxfp4_quant_image:
 *   a_bf16  : bf16 [m, k], row stride lda elements
 *   a_image : u8 [a_image_bytes], opaque; valid only for this (m, k).  The
 *             padding rows of its last 128-row tile are left as they were.
 * Preconditions: m > 0, k > 0, k % 32 == 0, lda >= k, lda % 8 == 0,
 * a_image_bytes >= mxfp4_act_image_bytes(m, k), a_bf16 and a_image 16-byte
 * aligned.  Errors: MXFP4_ERR_INVALID_ARG, MXFP4_ERR_CUDA.
 *
 * mxfp4_gemm_image: C[m,n] = bf16( A_image . B^T ) exactly as mxfp4_gemm
 * computes it from the A the image was made of (the same quantized values;
 * the summation order may differ from mxfp4_gemm's for m <= 32, which
 * quantizes inside its own kernel).  Needs no workspace.  The image may be
 * written by the kernel launched just before on the same stream
 * (mxfp4_quant_image): the GEMM waits for that kernel before reading it.
 * Preconditions: as mxfp4_gemm, with a_image from mxfp4_quant_image(m, k)
 * and 16-byte aligned.  Errors: MXFP4_ERR_INVALID_ARG,
 * MXFP4_ERR_UNSUPPORTED, MXFP4_ERR_CUDA.
 */
MXFP4_API size_t mxfp4_act_image_bytes(int64_t m, int64_t k);
MXFP4_API mxfp4_status mxfp4_quant_image(const void* a_bf16, int64_t m, int64_t k, int64_t lda, void* a_image,
                                         size_t a_image_bytes, void* stream);
MXFP4_API mxfp4_status mxfp4_gemm_image(const void* a_image, int64_t m, int64_t k, const void* b_packed, int64_t n,
                                        void* c_bf16, int64_t ldc, void* stream);

/*
 * Size of the scratch array built into the library for mxfp4_gemm_noalloc.
 */
#define MXFP4_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * mxfp4_gemm_noalloc -- the same operation, arguments and results as
 * mxfp4_gemm, for callers that cannot allocate device memory or pass a
 * workspace (for example a plugin whose host interface has no scratch
 * argument, or an engine that has committed all device memory up front).
 * The pages have no counterpart to this entry point.
 *   Scratch: a device array of MXFP4_NOALLOC_SCRATCH_BYTES (8 MiB) inside
 *   the library, held by every device that loads it until process exit.
 *   The call allocates nothing.  A shape that needs more scratch than that
 *   (mxfp4_gemm_workspace_bytes(m, n, k) > MXFP4_NOALLOC_SCRATCH_BYTES) is
 *   rejected with MXFP4_ERR_WORKSPACE before anything is enqueued.
 *   The first call on a device that needs scratch looks up the array's
 *   device address with that device current and keeps it (a failed lookup
 *   is not kept: the next call tries again); make that first call before
 *   any stream capture.
 *   All calls on a device share the one array: calls that may overlap on
 *   the GPU (unordered streams) race; calls ordered in one stream do not.
 *   Each call rewrites the scratch it uses; nothing needs to start at zero.
 */
MXFP4_API mxfp4_status mxfp4_gemm_noalloc(const void* a_bf16, int64_t m, int64_t k, int64_t lda,
                                          const void* b_packed, int64_t n, void* c_bf16, int64_t ldc,
                                          void* stream);

/*
 * mxfp4_measure_fp4_peak -- the dense block-scaled FP4 tensor-core rate of
 * the current device, in TFLOP/s, for roofline fractions: one CTA per SM
 * issues kblocks_per_sm back-to-back 128 x 256 x 256 K blocks of
 * tcgen05.mma kind::mxf4 (the GEMM kernels' issue sequence) on operands held
 * in shared memory, and the launch is timed with CUDA events on `stream`.
 * The pages quote no FP4 peak for this hardware; NVIDIA's nominal dense
 * figure for GB300 is 13.5 PFLOP/s.
 *   kblocks_per_sm: 1 .. 2^24 (about 2000 gives a launch of ~1 ms)
 *   tflops        : out, FLOPs (2 * 128 * 256 * 256 per K block and SM) / time
 * Blocks the host until the launch has finished (a measurement, not a
 * pipeline step).  Errors: MXFP4_ERR_INVALID_ARG, MXFP4_ERR_CUDA,
 * MXFP4_ERR_TIMEOUT (the bounded completion wait ran out).
 */
MXFP4_API mxfp4_status mxfp4_measure_fp4_peak(int64_t kblocks_per_sm, double* tflops, void* stream);

/*
 * mxfp4_launch_empty -- enqueue `count` (1..16) empty kernels of `ctas`
 * (1..65535) 32-thread CTAs on `stream`: the launch floor the small-m GEMM
 * (one launch, latency-bound) is measured against with the same event
 * method.  Errors: MXFP4_ERR_INVALID_ARG, MXFP4_ERR_CUDA.
 */
MXFP4_API mxfp4_status mxfp4_launch_empty(int count, int ctas, void* stream);

/*
 * mxfp4_launch_minimal -- enqueue `count` (1..16) minimal kernels of `ctas`
 * (1..65535) 32-thread CTAs on `stream`: each CTA reads one word of a
 * library-owned device array, allocates and frees 32 tensor-memory columns
 * and writes one word of the same array.  That is the least any GEMM launch
 * does; after an L2 flush by writes, any one of the three adds about 2 us
 * of event time to an empty kernel on GB300 (all three together the same),
 * so this is the floor a tcgen05 GEMM can meet.  Overlapping calls race on the
 * array, harmlessly (its values are never read by anything else).
 * Errors: MXFP4_ERR_INVALID_ARG, MXFP4_ERR_CUDA.
 */
MXFP4_API mxfp4_status mxfp4_launch_minimal(int count, int ctas, void* stream);

/*
 * mxfp4_set_debug_options -- testing and tuning overrides, process-wide,
 * for every later call on any thread: split_k forces the number of CTAs the
 * small-m GEMMs split K over (0 = the planner's own choice, else 1 to 8,
 * reduced where the shape or the cluster residency does not allow it);
 * drop_copies = 1 makes the GEMM kernels skip their operand copies (the
 * large-m kernel: forward no "stage landed" between the CTAs of a pair), so
 * that their bounded waits run out and the watchdog flag is raised: the
 * failure-detection path of mxfp4_device_status, exercised without any GPU
 * fault.  The initial values come from the environment variables
 * MXFP4_SPLIT_K and MXFP4_DEBUG_DROP_COPIES=1, read once when the library is
 * loaded.  The pages have no counterpart.  Errors: MXFP4_ERR_INVALID_ARG for
 * values outside those sets (nothing is changed).
 */
MXFP4_API mxfp4_status mxfp4_set_debug_options(int split_k, int drop_copies);

/*
 * mxfp4_kernel_binary_version -- the binaryVersion (major * 10 + minor) of
 * the library's GEMM kernel as loaded on the current device: 103 for the
 * sm_103a code this library is built with.  A diagnostic of the build; the
 * pages have no counterpart.  Errors: MXFP4_ERR_INVALID_ARG (null version),
 * MXFP4_ERR_CUDA (the query failed, e.g. no usable device).
 */
MXFP4_API mxfp4_status mxfp4_kernel_binary_version(int* version);

/*
 * mxfp4_device_status -- synchronize `stream`, then report and clear the
 * device-side watchdog flag: MXFP4_ERR_TIMEOUT if any kernel of this
 * library on the current device gave up a bounded pipeline wait since the
 * last call, MXFP4_ERR_CUDA if the synchronization failed, else MXFP4_OK.
 * This is a diagnostic call; it blocks the host.
 */
MXFP4_API mxfp4_status mxfp4_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_H_ */
