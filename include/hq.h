/*
 * hq.h -- C ABI of libhq: fused Hadamard rotation + NVFP4 quantization on GB300 (sm_103a).
 *
 * What is computed ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §1 "The format,
 * precisely" and §2 "The kernel"; storage layout from "NVFP4 Quantization" (Atlas docs),
 * "The numeric format"):
 *
 *   x       : M x K activations, row-major, row stride ldx elements (ldx >= K).
 *   rotation: every run of G consecutive elements of a row is multiplied by the
 *             Sylvester-Hadamard matrix H_G scaled by 1/sqrt(G):  y = x . H_G / sqrt(G).
 *             G = 16, G = 256 (= H16 (x) H16, scaled by 1/16), or G = 0 (rotation off: y = x).
 *             Computed as a fixed-order fp32 butterfly: stages h = 1, 2, 4, ..., G/2, each
 *             (a, b) -> (a + b, a - b), then one multiply by 1/sqrt(G).
 *   amax    : max |y| over the whole tensor (exact).
 *   s_global: amax / (448 * 6) in one fp32 division; 1.0 if that quotient is 0.
 *   blocks  : every 16 consecutive elements of a row of y form one NVFP4 block.
 *   s_block : E4M3 (float8 e4m3fn) value nearest to (block_amax / 6) / s_global, ties to even,
 *             saturating at 448.  Stored as its 8-bit pattern.
 *   codes   : s_f = s_block * s_global; if s_f == 0 every code of the block is 0, otherwise
 *             code = E2M1 value nearest to y / s_f (IEEE fp32 division), grid
 *             {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, saturating at 6; bit 3 copies
 *             the sign bit of the quotient (so -0.0 encodes as 0x8).
 *   packing : q[r][j] = code[r][2j] | (code[r][2j+1] << 4)   (even element in the low nibble).
 *
 * Layouts (all row-major, contiguous, owned by the caller):
 *   q       : uint8 [M, K/2]
 *   scales  : uint8 [M, K/16]  (E4M3 bit patterns)
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller.  The library allocates no memory,
 *     creates no stream and never synchronises the host; all work is enqueued on `stream`
 *     (a cudaStream_t / CUstream of the current device; NULL = the legacy default stream).
 *   - Argument errors are detected on the host before anything is enqueued and are returned
 *     synchronously; nothing is launched in that case.
 *   - A failed launch returns HQ_ERR_CUDA; hq_last_cuda_error() then gives the cudaError_t.
 *   - An empty tensor (M == 0 or K == 0, with valid sizes) is a no-op that returns HQ_OK; its
 *     data pointers may be NULL.  hq_rot_amax still writes 0 to `amax`, which must be valid.
 *   - Non-finite input is outside the contract.  hq_rot_amax reports it: a NaN anywhere gives
 *     a NaN amax and an infinity gives +inf, which the caller can read back.  Codes and scales
 *     for such tensors are unspecified.  Nothing traps or waits on the device.
 *   - Sizes are 64-bit element counts.
 */
#ifndef HQ_H_
#define HQ_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HQ_API __attribute__((visibility("default")))
#else
#define HQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HQ_OK = 0,
  HQ_ERR_NULL = 1,  /* a required pointer is NULL */
  HQ_ERR_SHAPE = 2, /* M < 0, K < 0, ldx < K, K not a multiple of max(16, G), M * K beyond
                       int64, or, in the calls that read x, K >= 2^36 (a row of 2^32 or
                       more 16-element blocks) */
  HQ_ERR_ALIGN = 3, /* a pointer or the row stride breaks the alignment rules below */
  HQ_ERR_DTYPE = 4, /* unknown element type */
  HQ_ERR_GROUP = 5, /* rotation group not in {0, 16, 256} */
  HQ_ERR_CUDA = 6,  /* the CUDA runtime refused a launch or an enqueue */
  HQ_ERR_TOO_LARGE = 7, /* the tensor does not fit the fixed scratch of
                           hq_quantize_nvfp4_host_noalloc */
  HQ_ERR_ALIAS = 8      /* two buffers that must be distinct are the same */
} hq_status;

typedef enum {
  HQ_F32 = 0, /* IEEE binary32 */
  HQ_BF16 = 1 /* bfloat16; widened to fp32 exactly */
} hq_dtype;

/* A cudaStream_t (CUstream) passed as a plain pointer. */
typedef void* hq_stream;

/*
 * hq_rot_amax -- pass 1: rotate and reduce the global amax.
 *   ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §2, "The global scale is the one
 *    thing not fused": the amax of the whole rotated tensor is needed before any block scale.)
 *
 *   x      : [M, K] of `dtype`, row stride ldx elements.  16-byte aligned; ldx * sizeof(dtype)
 *            a multiple of 16 bytes.
 *   group  : 0, 16 or 256.  K must be a multiple of max(16, group).
 *   amax   : 1 float, overwritten with max |y| (this call zeroes it first, on `stream`).
 *            4-byte aligned.
 *   y      : optional fp32 [M, K] (row stride K), 16-byte aligned, receives the rotated tensor;
 *            NULL to skip (the normal case: the rotation is never stored).
 */
HQ_API hq_status hq_rot_amax(const void* x, hq_dtype dtype, int64_t M, int64_t K, int64_t ldx,
                      int group, float* amax, float* y, hq_stream stream);

/*
 * hq_rotate_quant_nvfp4 -- pass 2: one read of x, one write of the codes and block scales.
 *   ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §1 table and §2 kernel: rotate,
 *    block amax, E4M3 scale, E2M1 codes, two codes per byte.)
 *
 *   x, dtype, M, K, ldx, group : as for hq_rot_amax.
 *   amax     : 1 float on the device, the global amax of the rotated tensor (normally written by
 *              hq_rot_amax on the same stream; any non-negative finite value is accepted, e.g.
 *              an amax kept from an earlier step).
 *   q        : uint8 [M, K/2], 16-byte aligned.
 *   scales   : uint8 [M, K/16], 4-byte aligned.
 *   s_global : optional 1 float, receives s_global (the per-tensor fp32 scale); NULL to skip.
 */
HQ_API hq_status hq_rotate_quant_nvfp4(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                int64_t ldx, int group, const float* amax, uint8_t* q,
                                uint8_t* scales, float* s_global, hq_stream stream);

/* Size of the workspace of hq_quantize_nvfp4 and the _ws entry points (hq_rotate_quant_nvfp4_ws,
 * hq_rotate_quant_nvfp4_swizzled_ws, hq_rotate_quant_nvfp4_delayed_ws, hq_rotate_quant_mxfp4_ws),
 * in 32-bit words
 * (control words and the counters of the run-time tile schedule, each on its own 128-byte
 * line). */
#define HQ_QUANTIZE_WORKSPACE_WORDS 288

/*
 * hq_quantize_nvfp4 -- both passes in one call: *amax, then codes, scales and s_global exactly as
 *   hq_rot_amax followed by hq_rotate_quant_nvfp4 on the same stream.
 *   ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §2: the global scale needs the
 *    amax of the whole rotated tensor before any block is quantized, hence two passes over x.)
 *
 *   Two launches, pass 1 then pass 2.  With `workspace`, pass 1 reduces the amax into the
 *   workspace and its last CTA writes *amax (no memset before it); pass 2 is
 *   hq_rotate_quant_nvfp4_ws (tiles handed out at run time) and fetches its first tiles of x
 *   while pass 1 ends; both launches are programmatic dependents of the kernel before them on
 *   the stream (each waits for that kernel to complete before it reads what the kernel
 *   wrote).  Without, pass 1 is hq_rot_amax and pass 2 hq_rotate_quant_nvfp4.
 *
 *   x, dtype, M, K, ldx, group : as for hq_rot_amax.
 *   amax      : 1 float on the device (written; 0 for an empty tensor).
 *   q, scales, s_global : as for hq_rotate_quant_nvfp4.
 *   workspace : NULL (hq_rot_amax then hq_rotate_quant_nvfp4), or HQ_QUANTIZE_WORKSPACE_WORDS
 *               uint32 on the device, 4-byte aligned, all 0 before its first use (e.g.
 *               cudaMemset).  Each call that records no fault leaves it 0 again.  Calls that may
 *               run at the same time (different streams) need different workspaces.
 */
HQ_API hq_status hq_quantize_nvfp4(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                   int64_t ldx, int group, float* amax, uint8_t* q,
                                   uint8_t* scales, float* s_global, uint32_t* workspace,
                                   hq_stream stream);

/*
 * hq_rotate_quant_nvfp4_ws -- pass 2 exactly as hq_rotate_quant_nvfp4 (same arguments, same
 *   outputs), with the tiles of x handed to the warps at run time instead of by a fixed split.
 *   (Not a step of the pages' method: a schedule.  With a fixed split the warps of an SM
 *   advance at different speeds, and the last ones still run while the others have left,
 *   with the memory system part idle.  Here each warp takes its next tile from a counter in
 *   `workspace`, so all warps run out of work at about the same time.)
 *
 *   workspace : HQ_QUANTIZE_WORKSPACE_WORDS uint32 on the device, 4-byte aligned, all 0 before
 *               its first use (e.g. cudaMemset); each call that records no fault leaves it 0
 *               again.  Calls that may run at the same time (different streams) need different
 *               workspaces; hq_quantize_nvfp4's may be shared with it on one stream.
 *               NULL: the fixed split of hq_rotate_quant_nvfp4.
 */
HQ_API hq_status hq_rotate_quant_nvfp4_ws(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                          int64_t ldx, int group, const float* amax, uint8_t* q,
                                          uint8_t* scales, float* s_global, uint32_t* workspace,
                                          hq_stream stream);

/*
 * hq_rotate_quant_nvfp4_swizzled -- pass 2 exactly as hq_rotate_quant_nvfp4, with the E4M3 block
 * scales written straight into the tiled layout that block-scaled NVFP4 GEMMs read.
 *   ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §6 "From interpreter to
 *    hardware", Layout: cuBLASLt and CUTLASS take the block scales in a swizzled tiled layout,
 *    and a production kernel writes it directly; the page does not spell the layout out.  The
 *    layout here is cuBLASLt's for 16-element block scales; the GPU tests check it by feeding
 *    the output to cuBLASLt's NVFP4 GEMM.)
 *
 *   scales : hq_swizzled_scales_bytes(M, K) bytes, 32-byte aligned.  The [M, K/16] scale
 *            matrix is padded to R = round_up(M, 128) rows and C = round_up(K/16, 4) columns
 *            and cut into tiles of 128 rows x 4 columns; tile (i, j) is the 512 bytes at
 *            (i * C/4 + j) * 512, and inside it row r, column c (r < 128, c < 4) is the byte
 *            (r % 32) * 16 + (r / 32) * 4 + c.  Every byte is written, padding entries as 0
 *            (a GEMM reads them).
 *   Everything else (x, amax, q, s_global, group, errors) as hq_rotate_quant_nvfp4.
 */
HQ_API hq_status hq_rotate_quant_nvfp4_swizzled(const void* x, hq_dtype dtype, int64_t M,
                                                int64_t K, int64_t ldx, int group,
                                                const float* amax, uint8_t* q, uint8_t* scales,
                                                float* s_global, hq_stream stream);

/*
 * hq_rotate_quant_nvfp4_swizzled_ws -- hq_rotate_quant_nvfp4_swizzled exactly (same arguments,
 *   same outputs), with its units of work (8 rows x 128 blocks) handed to the warps at run time
 *   as in hq_rotate_quant_nvfp4_ws (a schedule, not a step of the method).
 *   workspace : as for hq_rotate_quant_nvfp4_ws.  NULL: hq_rotate_quant_nvfp4_swizzled.
 */
HQ_API hq_status hq_rotate_quant_nvfp4_swizzled_ws(const void* x, hq_dtype dtype, int64_t M,
                                                   int64_t K, int64_t ldx, int group,
                                                   const float* amax, uint8_t* q,
                                                   uint8_t* scales, float* s_global,
                                                   uint32_t* workspace, hq_stream stream);

/* Size in bytes of the swizzled scale buffer for an [M, K] tensor (-1 if M < 0, K < 0,
 * K % 16 != 0, or the size does not fit int64). */
HQ_API int64_t hq_swizzled_scales_bytes(int64_t M, int64_t K);

/*
 * hq_rotate_quant_nvfp4_delayed -- single-pass mode: quantize with an amax kept from an earlier
 *   step while reducing this tensor's amax for the next one.
 *   ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §2, on the global scale:
 *    production stacks run a small amax reduction ahead of the kernel *or reuse an amax from a
 *    previous step*, so that the per-block work stays a single pass.)
 *
 *   Reads x once.  Codes, scales and s_global are exactly those of hq_rotate_quant_nvfp4 with
 *   amax = *amax_prev; *amax_next receives max |y| of this tensor, exactly as hq_rot_amax would
 *   (this call zeroes it first, on `stream`).  When *amax_prev is smaller than this tensor's
 *   amax, blocks whose scale would exceed 448 saturate (scale 448, codes clipped at 6): the
 *   price of a stale global scale.
 *
 *   x, dtype, M, K, ldx, group, q, scales, s_global : as for hq_rotate_quant_nvfp4.
 *   amax_prev : 1 float on the device (read).      amax_next : 1 float on the device (written).
 *   The two must be different floats; passing the same pointer returns HQ_ERR_ALIAS.
 */
HQ_API hq_status hq_rotate_quant_nvfp4_delayed(const void* x, hq_dtype dtype, int64_t M,
                                               int64_t K, int64_t ldx, int group,
                                               const float* amax_prev, float* amax_next,
                                               uint8_t* q, uint8_t* scales, float* s_global,
                                               hq_stream stream);

/*
 * hq_rotate_quant_nvfp4_delayed_ws -- hq_rotate_quant_nvfp4_delayed exactly (same arguments, same
 *   outputs), with a workspace: the tiles of x are handed to the warps at run time as in
 *   hq_rotate_quant_nvfp4_ws, and *amax_next is reduced in the workspace and written by the
 *   kernel's last CTA, so no memset runs before it (one launch per call).
 *   workspace : as for hq_rotate_quant_nvfp4_ws.  NULL: hq_rotate_quant_nvfp4_delayed.
 */
HQ_API hq_status hq_rotate_quant_nvfp4_delayed_ws(const void* x, hq_dtype dtype, int64_t M,
                                                  int64_t K, int64_t ldx, int group,
                                                  const float* amax_prev, float* amax_next,
                                                  uint8_t* q, uint8_t* scales, float* s_global,
                                                  uint32_t* workspace, hq_stream stream);

/*
 * hq_rotate_quant_mxfp4 -- MXFP4 variant: E2M1 codes with one power-of-two (E8M0) scale per 32
 *   consecutive elements of a row and no per-tensor scale, so a single pass over x.
 *   ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §1: MXFP4 has 32-element blocks and
 *    power-of-two E8M0 scales; "Try this": the error study with MXFP4 semantics.)
 *   The pages give no rule for the scale; this library uses the usual MX rule:
 *   X = 2^(floor(log2 amax_32) - 2), so amax_32 / X lies in [4, 8) (2 is the exponent of E2M1's
 *   largest value, 6); the stored byte is the exponent + 127, clamped to [0, 254] (0 for an
 *   all-zero block); codes = E2M1(y / X) as for NVFP4 (ties to even, saturating at 6, sign bit
 *   copied).  The rotation is as for NVFP4 (group 0, 16 or 256).
 *
 *   x, dtype, M, K, ldx, group : as for hq_rotate_quant_nvfp4, with K a multiple of 32 as well.
 *   q      : uint8 [M, K/2], 16-byte aligned (same packing as NVFP4).
 *   scales : uint8 [M, K/32] E8M0 bytes.
 */
HQ_API hq_status hq_rotate_quant_mxfp4(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                       int64_t ldx, int group, uint8_t* q, uint8_t* scales,
                                       hq_stream stream);

/*
 * hq_rotate_quant_mxfp4_ws -- hq_rotate_quant_mxfp4 exactly (same arguments, same outputs), with
 *   the tiles of x handed to the warps at run time as in hq_rotate_quant_nvfp4_ws (a schedule,
 *   not a step of the method).
 *   workspace : as for hq_rotate_quant_nvfp4_ws (HQ_QUANTIZE_WORKSPACE_WORDS uint32, all 0
 *               before its first use and left 0 by each call that records no fault; one per
 *               stream that may run at the same time).  NULL: hq_rotate_quant_mxfp4.
 */
HQ_API hq_status hq_rotate_quant_mxfp4_ws(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                          int64_t ldx, int group, uint8_t* q, uint8_t* scales,
                                          uint32_t* workspace, hq_stream stream);

/* hq_dequant_mxfp4 -- value = (+-grid[code & 7]) * 2^(byte - 127), then the rotation again when
 * `unrotate` (group 16 or 256).  out: fp32 [M, K], 16-byte aligned; q 8-byte aligned. */
HQ_API hq_status hq_dequant_mxfp4(const uint8_t* q, const uint8_t* scales, int64_t M, int64_t K,
                                  int group, int unrotate, float* out, hq_stream stream);

/*
 * hq_rotate_quant_int8 -- INT8 per-token rotate-quant with the regular Hadamard.
 *   ("hyperflow_h3_flash_int8.py", HyperFlow: regular_hadamard, rotate_quant_kernel; the
 *    activation side of a W8A8 linear whose weight was rotated offline.)
 *
 *   y      = x . R_G on every run of G consecutive channels of a row, R_G = kron(H4/2, ...)
 *            (log4 G factors), H4 = [[1,1,1,-1],[1,1,-1,1],[1,-1,1,1],[-1,1,1,1]] (orthonormal,
 *            symmetric, rows summing to one).  Fixed fp32 order: the base-4 digits of the
 *            channel index from the least significant, each 4-point step out_k = RN(S/2 -
 *            v_(3-k)), S = (v0 + v1) + (v2 + v3).  (The page's group of 1024 is computed from
 *            its 16 x 64 factors; the Kronecker power is the same matrix, and the digit order
 *            fixes the rounding.)
 *   scales : fp32 [M], scale = max(amax_row |y|, 1e-12) / 127.
 *   q      : int8 [M, K] row-major, q = clamp(rint(y * (1/scale)), -127, 127) (half to even).
 *   For K <= 120832, x is read once and the rotated row stays on chip until its amax is known
 *   (tensor memory up to 32768 channels, tensor and shared memory beyond); a longer row is read
 *   twice, first for its amax and then to quantize it (the second read mostly from L2).
 *
 *   group  : 4, 16, 64, 256 or 1024; K a multiple of the group and of 16 (the kernels move
 *            whole 16-channel blocks), K / 2048 below 2^30.
 *   x      : [M, K] of dtype, row stride ldx (16-byte aligned; ldx * sizeof(dtype) % 16 == 0).
 *   q      : 16-byte aligned.   scales : 4-byte aligned.
 */
HQ_API hq_status hq_rotate_quant_int8(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                      int64_t ldx, int group, int8_t* q, float* scales,
                                      hq_stream stream);

/*
 * hq_dequant_nvfp4 -- round trip for checks (not part of the quantization hot path).
 *   ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §2 dequantize:
 *    value = (+-grid[code & 7]) * (s_block * s_global), then the rotation applied again when the
 *    data was rotated; H_G / sqrt(G) is symmetric and orthonormal, so it is its own inverse.)
 *
 *   q, scales : as written by hq_rotate_quant_nvfp4 (q 8-byte aligned).
 *   s_global  : 1 float on the device.
 *   group     : 0, 16 or 256; the rotation to undo when `unrotate` is non-zero (then 16 or 256,
 *               and K a multiple of it); otherwise only checked.
 *   out       : fp32 [M, K] (row stride K), 16-byte aligned.
 *   The two products are rounded in that order (s_f first), then the butterfly as above.
 */
HQ_API hq_status hq_dequant_nvfp4(const uint8_t* q, const uint8_t* scales, const float* s_global,
                           int64_t M, int64_t K, int group, int unrotate, float* out,
                           hq_stream stream);

/* Human-readable name of a status code (static storage). */
HQ_API const char* hq_status_string(hq_status status);

/* The cudaError_t behind the last HQ_ERR_CUDA returned on the calling host thread (0 if none). */
HQ_API int hq_last_cuda_error(void);

/*
 * hq_read_fault -- the library's device fault word on the current device (synchronous: waits
 * for all work on the device first).  0 means no kernel recorded a fault.  Bit 0 (value 1):
 * a kernel's wait for one of its own shared-memory tile copies exceeded about one second; that
 * warp stopped early, so the outputs of the affected call are incomplete.  With `clear` non-zero
 * the word is reset to 0 after reading.
 */
HQ_API hq_status hq_read_fault(unsigned int* fault, int clear);

/*
 * hq_selftest_bounded_wait -- a test of the failure detection above, not part of the
 * quantization path (the pages have no counterpart).  Launches one warp on `stream` that waits,
 * through the same bounded mbarrier wait as the kernels' tile pipelines, on a barrier that nothing
 * ever completes.  After about one second the wait gives up, the kernel sets bit 0 of the fault
 * word and returns; no memory is touched and the context stays usable.  Returns once the launch
 * is enqueued (read the result with hq_read_fault).
 *   unit : 0 runs the wait in the translation unit of the NVFP4 / MXFP4 kernels, 1 in that of
 *          the INT8 kernel (each has its own copy of the fault word; hq_read_fault reads both).
 *          Anything else: HQ_ERR_SHAPE.
 */
HQ_API hq_status hq_selftest_bounded_wait(int unit, hq_stream stream);

/*
 * Host pipeline -- quantize tensors that live in (pinned) host memory.
 *   Not a step of the method itself: the transport around it.  One submission copies x to the
 *   device, runs hq_rot_amax and hq_rotate_quant_nvfp4 there, and moves the codes, the scales
 *   and s_global back.  Consecutive submissions overlap: the pipeline alternates between two
 *   buffer sets in the caller's device workspace and runs input copies, kernels and output
 *   transfers on three streams of its own, ordered by events, so the input copy of one
 *   submission runs while the previous one computes and sends its results back.  The outputs
 *   are written into the host buffers by a small kernel when the device can address them
 *   (pinned or registered memory, or any host memory on a device that reaches pageable memory
 *   through the host page tables), and copied otherwise.
 *
 *   The pipeline object is host memory owned by the library (freed by _destroy); it also owns
 *   three CUDA streams and six events on the device that is current at _create.  It allocates
 *   no device memory: `d_work` (at least hq_host_pipeline_workspace_bytes(M, K, dtype) bytes,
 *   256-byte aligned, owned by the caller) holds both buffer sets.  Host buffers should be pinned
 *   (cudaHostAlloc / cudaHostRegister) for the copies to be asynchronous; every host buffer of a
 *   submission must stay valid and untouched until hq_host_pipeline_wait() returns.
 */
typedef struct hq_host_pipeline hq_host_pipeline;

/* Device workspace bytes for M x K tensors of `dtype`.  0 if the sizes are invalid: M or K not
 * positive, K not a multiple of 16, K >= 2^36, or more than 2^58 elements. */
HQ_API size_t hq_host_pipeline_workspace_bytes(int64_t M, int64_t K, hq_dtype dtype);

/* Create a pipeline for M x K row-major tensors (contiguous rows) and rotation `group`. */
HQ_API hq_status hq_host_pipeline_create(int64_t M, int64_t K, hq_dtype dtype, int group,
                                         void* d_work, size_t work_bytes,
                                         hq_host_pipeline** out);

/* Enqueue one quantization and return at once.  x_host: [M, K] of dtype; q_host: [M, K/2] bytes;
 * scales_host: [M, K/16] bytes; s_global_host: 1 float.  Results are complete after
 * hq_host_pipeline_wait().
 * If a step fails after part of the submission was enqueued (HQ_ERR_CUDA), the buffer set's
 * ordering events may not cover the work in flight, so the pipeline refuses every later
 * submission with HQ_ERR_CUDA (hq_last_cuda_error() gives the first failure); wait for it and
 * destroy it.  A submission refused before anything was enqueued (HQ_ERR_NULL) leaves it usable. */
HQ_API hq_status hq_host_pipeline_submit(hq_host_pipeline* p, const void* x_host, uint8_t* q_host,
                                         uint8_t* scales_host, float* s_global_host);

/* Block the calling thread until every submitted quantization has finished. */
HQ_API hq_status hq_host_pipeline_wait(hq_host_pipeline* p);

/* Wait for outstanding work, then release the streams, events and the object (NULL is a no-op). */
HQ_API hq_status hq_host_pipeline_destroy(hq_host_pipeline* p);

/* hq_host_pipeline_inject_failure -- a test of the failure handling above, not part of the
 * quantization path (the pages have no counterpart).  The next submission to `p` behaves as if
 * the CUDA runtime refused its step `step` (0 the input copy, 1 pass 1, 2 pass 2, 3 the output
 * transfer): that step and the ones after it are not enqueued, the submission returns
 * HQ_ERR_CUDA with cudaErrorNotPermitted recorded, and the steps before it stay enqueued.
 * Nothing on the device fails.  step < 0 cancels a pending injection; step > 3: HQ_ERR_SHAPE. */
HQ_API hq_status hq_host_pipeline_inject_failure(hq_host_pipeline* p, int step);

/*
 * hq_quantize_nvfp4_host_noalloc -- the quantization of one host tensor with no device
 * allocation at all.  The pages have no counterpart: this entry point is for callers that cannot
 * obtain device memory themselves.  Examples: a plug-in loaded into a host program that owns the
 * whole device memory pool and hands its extensions no allocator; a serving loop that fixed its
 * memory footprint at start-up and must not allocate on the request path (an allocation there
 * can fail, or stall on the allocator).  Those callers can neither provide the workspace of the
 * host pipeline nor let the library allocate one.
 *
 * It does what one submission of the host pipeline does, in order on `stream`: copy x_host to the
 * device, hq_rot_amax, hq_rotate_quant_nvfp4, copy the codes, scales and s_global back.  Results
 * are complete when `stream` reaches that point (synchronize it, or record an event).  Its
 * device staging is one fixed array of HQ_NOALLOC_SCRATCH_BYTES inside the library, reserved on
 * every device where the library is loaded and held until the process exits.
 *
 *   Limit: the tensor must fit that array: with n = M*K and e = 2 (bf16) or 4 (fp32) bytes,
 *   r(b) = b rounded up to a multiple of 256, it needs r(n e) + r(n/2) + r(n/16) + 512 bytes
 *   (about 13.1 million bf16 or 7.35 million fp32 elements).  Larger tensors return
 *   HQ_ERR_TOO_LARGE before anything is enqueued.
 *   Set-up: the first call on a device looks up the array's device address (once per device,
 *   with that device current), so make that first call before any stream capture.  The address
 *   belongs to the device's context: after cudaDeviceReset the next call looks it up again (and
 *   is then a first call again).
 *   Sharing: every call on a device uses the same array and leaves its contents there; calls
 *   whose work overlaps on the GPU (other streams, other host threads) race on it, so order
 *   them (one stream, or events).  The call clears what must start at zero (the amax).
 *   Host buffers should be pinned for the copies to be asynchronous.  x_host: [M, K] of dtype,
 *   contiguous rows; q_host: [M, K/2]; scales_host: [M, K/16]; s_global_host: 1 float.
 */
#define HQ_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
HQ_API hq_status hq_quantize_nvfp4_host_noalloc(const void* x_host, hq_dtype dtype, int64_t M,
                                                int64_t K, int group, uint8_t* q_host,
                                                uint8_t* scales_host, float* s_global_host,
                                                hq_stream stream);

/* Library version: major * 10000 + minor * 100 + patch. */
HQ_API int hq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HQ_H_ */
