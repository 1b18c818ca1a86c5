/*
 * fp4codec.h -- C ABI of the block-scaled FP4 (E2M1) codec for GB300 (sm_103a).
 *
 * Sources (cited by short key below):
 *   [FP4Quant]  cybernoise.de, "FP4Quant speeds up GPU communication, with a
 *               measurable accuracy trade-off".
 *   [fp4-train] huggingface.co/kernels/phanerozoic/fp4-train, model card.
 *   [MoE-FP4]   paper-daily.com review (2026-03-05) of "Practical FP4 Training
 *               for Large-Scale MoE Models on Hopper GPUs".
 *   [WP2]       hiren.me, "Weight precision, part 2".
 *
 * Conventions, for every entry point:
 *   - Array pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or synchronizes.  Work is enqueued on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream) and is asynchronous.
 *   - Arguments are checked before anything is enqueued.  A failed check
 *     returns its status and enqueues nothing.  A launch error is returned as
 *     FP4_ERR_CUDA (the CUDA error is left for cudaGetLastError()).
 *   - Sizes are element counts.  A size of 0 is legal and enqueues nothing.
 *   - Packed E2M1 codes hold two codes per byte, element 2i in the low nibble;
 *     code bits: [3] sign, [2:1] exponent, [0] mantissa ([WP2] "What FP4 can
 *     hold"; [fp4-train] "How it works": the two-codes-per-byte layout).
 *   - Inputs must be finite.  NaN or infinite inputs give deterministic but
 *     unspecified codes.
 *   - The library keeps no state between calls except a process-wide count of
 *     kernel launches and the workspace of nvfp4_quantize_noalloc, so calls
 *     other than nvfp4_quantize_noalloc are thread-safe.
 */
#ifndef FP4CODEC_H
#define FP4CODEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP4CODEC_ABI_VERSION 1

typedef enum {
  FP4_OK = 0,
  FP4_ERR_NULL = 1,      /* a required pointer is NULL */
  FP4_ERR_ALIGN = 2,     /* a pointer breaks its stated alignment */
  FP4_ERR_SHAPE = 3,     /* a size is negative or breaks its divisibility rule */
  FP4_ERR_DTYPE = 4,     /* unknown dtype */
  FP4_ERR_ARG = 5,       /* another argument out of range (mode, group, ...) */
  FP4_ERR_CUDA = 6,      /* a kernel launch failed */
  FP4_ERR_INTERNAL = 7
} fp4_status;

typedef enum { FP4_F32 = 0, FP4_BF16 = 1 } fp4_dtype;
typedef enum { FP4_RTN = 0, FP4_SR = 1 } fp4_round;

/* How the NVFP4 per-tensor fp32 scale s_t is obtained ([WP2] "Block scaling":
 * one 32-bit scale for the whole matrix; the pages do not say how it is
 * chosen):
 *   GIVEN      read from *tensor_scale;
 *   COMPUTE    s_t = amax / (6 * 448) from a tensor-amax pass run inside the
 *              call (amax_ws is its workspace), written to *tensor_scale;
 *   FROM_AMAX  like COMPUTE, but the amax is the one a previous nvfp4_amax /
 *              nvfp4_qdq_amax call left in *amax_ws (no amax pass here).
 * In every mode a scale that is not finite or not > 0 is used as 1; COMPUTE
 * and FROM_AMAX write the scale they used, GIVEN never writes it. */
typedef enum { FP4_TSCALE_GIVEN = 0, FP4_TSCALE_COMPUTE = 1, FP4_TSCALE_FROM_AMAX = 2 } fp4_tscale;

const char* fp4_status_string(int status);
int fp4_abi_version(void);
/* Number of kernels this library has launched in this process. */
uint64_t fp4_kernel_launches(void);
/* Number of bounded waits in this library's kernels that gave up, on the
 * current device, since the library was loaded (the FP4Quant encode's waits
 * for its TMA copies).  0 in a healthy run; a warp that gives up skips the
 * rest of its work, so after a nonzero value the outputs of the launches
 * since the last read are not to be trusted.  Synchronizes with the device;
 * UINT64_MAX if the read fails. */
uint64_t fp4_wait_timeouts(void);
/* Test hook for the bounded waits: the bf16 G = 128 FP4Quant encode of x
 * [rows, cols] (cols % 128 == 0, at most 2^24 elements) with its TMA copies
 * announced 16 bytes longer than they are, so no wait completes: every warp
 * that has a tile gives up after its wait limit (about a second), adds 1 to
 * fp4_wait_timeouts() and returns without writing its outputs.  The context
 * stays usable.  Errors as fp4quant_encode. */
fp4_status fp4_test_encode_wait_timeout(const void* x, int64_t rows, int64_t cols,
                                        uint8_t* packed, float* s1, float* s2, void* stream);

/* ------------------------------------------------------------------ NVFP4
 * [fp4-train] "How it works": 16-element blocks, block scale block_absmax / 6
 * encoded to e4m3, every element divided by the decoded scale (e4m3 block
 * scale times s_t) and encoded to E2M1 by round-to-nearest-even or by
 * stochastic rounding from a counter-based (seed, step, global index) RNG,
 * optional per-element error-feedback residual.  "Requirements and limits":
 * float32 or bfloat16 input, K a multiple of 16.
 */

/* *amax_ws = max |x[i] (+ residual[i])| over n elements (NaN ignored).
 *   x         [n] fp32 or bf16, 32-byte aligned
 *   residual  [n] fp32, 32-byte aligned, or NULL
 *   amax_ws   1 fp32, 4-byte aligned; zeroed and then written by this call
 *   n % 16 == 0 */
fp4_status nvfp4_amax(const void* x, int dtype, int64_t n, const float* residual,
                      float* amax_ws, void* stream);

/* Quantize x (flat, n % 16 == 0) to NVFP4.
 *   x            [n] fp32 or bf16 (dtype), 32-byte aligned
 *   residual     [n] fp32 error-feedback residual, read and updated in place
 *                (r <- (x + r) - dequant(code)), 32-byte aligned, or NULL
 *   rounding     FP4_RTN or FP4_SR; SR draws a 16-bit uniform h per element
 *                from Philox4x32-10 with key = seed and counter = (g >> 3,
 *                step), g the flat element index: half g & 1 (low first) of
 *                word (g >> 1) & 3; the upper grid neighbour is taken iff
 *                h * 2^-16 < the fractional distance
 *   tscale_mode  fp4_tscale; tensor_scale: 1 fp32 on the device (read for
 *                GIVEN, written otherwise); amax_ws: 1 fp32 workspace, needed
 *                for COMPUTE and FROM_AMAX (may be NULL for GIVEN)
 *   packed       [n/2] bytes out, 16-byte aligned
 *   scales       [n/16] e4m3 bytes out, block b for elements 16b..16b+15,
 *                linear order (not swizzled) */
fp4_status nvfp4_quantize(const void* x, int dtype, int64_t n, float* residual,
                          int rounding, uint64_t seed, uint64_t step, int tscale_mode,
                          float* tensor_scale, float* amax_ws, uint8_t* packed,
                          uint8_t* scales, void* stream);

/* y[i] = value(code_i) * (e4m3(scales[i/16]) * s_t), one fp32 product,
 * then rounded to bf16 (nearest-even) if out_dtype is FP4_BF16.
 * ([WP2] "Block scaling", step 5: multiply back by the scale.)
 *   packed        [n/2], 16-byte aligned; scales [n/16], 2-byte aligned
 *   tensor_scale  1 fp32 on the device, or NULL for s_t = 1
 *   y             [n] out, 32-byte aligned; n % 16 == 0 */
fp4_status nvfp4_dequantize(const uint8_t* packed, const uint8_t* scales,
                            const float* tensor_scale, int64_t n, void* y, int out_dtype,
                            void* stream);

/* *amax_ws = max |(W - lr*G) + r| over n elements, for FROM_AMAX qdq. */
fp4_status nvfp4_qdq_amax(const uint16_t* w_bf16, const float* g, float lr,
                          const float* residual, int64_t n, float* amax_ws, void* stream);

/* One training step on an NVFP4-stored bf16 weight ([fp4-train] "Usage":
 * W = ef.qdq(key, W - lr * grad, step)):
 *   v = ((W - lr*G) + r), quantize v as nvfp4_quantize does, q = dequant,
 *   W <- bf16(q) in place, r <- v - q in place.
 *   w_bf16    [n] bf16, 32-byte aligned, updated in place
 *   g         [n] fp32 gradient, 32-byte aligned, or NULL (no update term)
 *   residual  [n] fp32, 32-byte aligned, or NULL (no error feedback)
 *   packed, scales  as nvfp4_quantize, or both NULL to skip writing them */
fp4_status nvfp4_qdq(uint16_t* w_bf16, const float* g, float lr, int64_t n, float* residual,
                     int rounding, uint64_t seed, uint64_t step, int tscale_mode,
                     float* tensor_scale, float* amax_ws, uint8_t* packed, uint8_t* scales,
                     void* stream);

/* nvfp4_quantize in COMPUTE mode without a caller-supplied workspace.  The
 * pages have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory: a plugin that is handed only the tensors it
 * works on by a framework or inference engine that owns all device memory,
 * or C code with no device allocator of its own.  Such callers cannot provide
 * the one-fp32 amax workspace that COMPUTE mode needs, so here that
 * workspace is a 256-byte array inside the library, in device memory that
 * every GPU which loads the library holds until the process exits.
 *   Arguments and results are those of nvfp4_quantize with
 *   tscale_mode = FP4_TSCALE_COMPUTE (tensor_scale is written).
 *   Scratch: one fp32 per call, whatever n is, out of a 256-byte array; a
 *   call whose scratch need exceeded the array would fail with
 *   FP4_ERR_SHAPE, which the one-fp32 need never does.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   The first call on each device looks the array's device address up with
 *   cudaGetSymbolAddress (with that device current) and caches it; make that
 *   first call before any stream capture on the device.  The cached address
 *   belongs to the device's context as it was at that first call: after a
 *   cudaDeviceReset (or any other reset of that context) in the same
 *   process it is stale, and the process must not call this entry point on
 *   that device again.
 *   Every call on a device shares the one slot, which the call clears before
 *   use; calls whose work overlaps on the GPU (other streams, or two host
 *   threads) race on it and must be serialized by the caller. */
fp4_status nvfp4_quantize_noalloc(const void* x, int dtype, int64_t n, float* residual,
                                  int rounding, uint64_t seed, uint64_t step,
                                  float* tensor_scale, uint8_t* packed, uint8_t* scales,
                                  void* stream);

/* ------------------------------------------------- blocked scale layout
 * [fp4-train] "Scope": the NVFP4 tensor-core matmul hands its e4m3 block
 * scales to the hardware after swizzling them into the layout
 * torch._scaled_mm consumes.  That layout ("blocked"): the [rows, cols]
 * one-byte scale matrix of a [rows, K] operand (cols = K/16 for NVFP4, K/32
 * for MXFP4) is zero-padded to [128 * ceil(rows/128), 4 * ceil(cols/4)], cut
 * into tiles of 128 rows x 4 columns stored in row-major tile order, 512
 * bytes each, and scale (r, c) of a tile sits at byte
 * 16 * (r % 32) + 4 * (r / 32) + c of its tile.
 */

/* Bytes of the blocked form of a [rows, cols] scale matrix, or -1 when
 * rows or cols is negative, either is >= 2^40, or the matrix has more than
 * 2^44 padded scales.  Host only; no device work. */
int64_t fp4_blocked_scales_size(int64_t rows, int64_t cols);

/* scales [rows, cols] row-major bytes (any alignment) -> blocked
 * [fp4_blocked_scales_size(rows, cols)] bytes, 16-byte aligned; every byte
 * of blocked is written, padding with 0.  Nothing to do for an empty
 * matrix.  The bytes are moved, not interpreted. */
fp4_status fp4_scales_to_blocked(const uint8_t* scales, int64_t rows, int64_t cols,
                                 uint8_t* blocked, void* stream);

/* The inverse: blocked (16-byte aligned) -> scales [rows, cols]; padding
 * bytes are ignored. */
fp4_status fp4_scales_from_blocked(const uint8_t* blocked, int64_t rows, int64_t cols,
                                   uint8_t* scales, void* stream);

/* nvfp4_quantize of a [rows, k] row-major matrix (k % 16 == 0, k < 2^28,
 * rows * k < 2^44) whose block scales are written straight into the blocked layout of
 * the [rows, k/16] scale matrix, padding included (no second pass).  Codes,
 * tensor scale, residual update and stochastic-rounding draws are those of
 * nvfp4_quantize on the flat n = rows * k elements, and blocked_scales equals
 * fp4_scales_to_blocked of nvfp4_quantize's scales.
 *   blocked_scales  [fp4_blocked_scales_size(rows, k/16)] bytes out, any
 *                   alignment; all other arguments as nvfp4_quantize. */
fp4_status nvfp4_quantize_blocked(const void* x, int dtype, int64_t rows, int64_t k,
                                  float* residual, int rounding, uint64_t seed, uint64_t step,
                                  int tscale_mode, float* tensor_scale, float* amax_ws,
                                  uint8_t* packed, uint8_t* blocked_scales, void* stream);

/* ------------------------------------------------------- NVFP4, batched
 * The same NVFP4 operations on a list of independent tensors in one launch
 * per pass (a whole model's weight matrices, say), each tensor with its own
 * per-tensor scale.  The result for every tensor is bit-identical to the
 * single-tensor call on it.  Each tensor is split into work chunks of
 * FP4_BATCH_CHUNK_BLOCKS 16-element blocks; the chunks of all tensors form
 * one flat index space that the kernels walk, so small tensors cost no
 * launch of their own.
 */
#define FP4_BATCH_CHUNK_BLOCKS 256

/* One tensor of a batch.  The array of these descriptors lives in device
 * memory (the caller fills it, e.g. by copying a host array prepared with
 * fp4_batch_plan).  Pointers are device pointers; fields an operation does
 * not use may be NULL (x for dequantize, y for amax/quantize). */
typedef struct {
  const void* x;        /* [n] input, fp32 or bf16, 32-byte aligned */
  uint8_t* packed;      /* [n/2] codes, 16-byte aligned */
  uint8_t* scales;      /* [n/16] e4m3 block scales, 2-byte aligned */
  void* y;              /* [n] dequantized output, 32-byte aligned */
  int64_t n;            /* elements, n % 16 == 0 (0 allowed), n < 2^44 */
  int64_t chunk_start;  /* index of the tensor's first chunk (fp4_batch_plan) */
} fp4_tensor_desc;

/* Host helper: checks every descriptor of a host array (n % 16, n < 2^44,
 * alignment of the non-NULL pointers) and count < 2^24 (FP4_ERR_SHAPE
 * otherwise), then fills chunk_start; *total_chunks receives the number of
 * chunks of the batch.  The batched calls trust a table that passed this
 * check. */
fp4_status fp4_batch_plan(fp4_tensor_desc* host_desc, int32_t count, int64_t* total_chunks);

/* amax[t] = max |x_t[i]| for every tensor t (as nvfp4_amax); amax is a
 * device array of count fp32 (4-byte aligned), zeroed and written. */
fp4_status nvfp4_amax_batched(const fp4_tensor_desc* desc, int32_t count, int64_t total_chunks,
                              int dtype, float* amax, void* stream);

/* nvfp4_quantize on every tensor (no error feedback): tensor_scale and amax
 * are device arrays of count fp32, read or written per tscale_mode exactly as
 * the single-tensor call does with its scalars; COMPUTE runs the batched
 * amax pass first.  Stochastic rounding draws with the element index inside
 * each tensor, as the single-tensor call does. */
fp4_status nvfp4_quantize_batched(const fp4_tensor_desc* desc, int32_t count, int64_t total_chunks,
                                  int dtype, int rounding, uint64_t seed, uint64_t step,
                                  int tscale_mode, float* tensor_scale, float* amax, void* stream);

/* nvfp4_quantize_batched with every tensor's block scales written in the
 * blocked layout of its [n_t / k_t, k_t] matrix, padding included (as
 * nvfp4_quantize_blocked does for one matrix): desc[t].scales points at
 * fp4_blocked_scales_size(n_t / k_t, k_t / 16) bytes (any alignment).
 *   k  device array of count int64, the row length k_t of each tensor,
 *      8-byte aligned; validated on the host by fp4_batch_plan_blocked.
 * Codes, tensor scales and SR draws are those of nvfp4_quantize_batched. */
fp4_status nvfp4_quantize_batched_blocked(const fp4_tensor_desc* desc, const int64_t* k,
                                          int32_t count, int64_t total_chunks, int dtype,
                                          int rounding, uint64_t seed, uint64_t step,
                                          int tscale_mode, float* tensor_scale, float* amax,
                                          void* stream);

/* Host helper: fp4_batch_plan plus, for every tensor, k_t > 0, k_t % 16 == 0,
 * k_t / 16 < 2^24 and n_t % k_t == 0 (FP4_ERR_SHAPE otherwise). */
fp4_status fp4_batch_plan_blocked(fp4_tensor_desc* host_desc, const int64_t* host_k, int32_t count,
                                  int64_t* total_chunks);

/* nvfp4_dequantize on every tensor; tensor_scale is a device array of count
 * fp32, or NULL for scale 1. */
fp4_status nvfp4_dequantize_batched(const fp4_tensor_desc* desc, int32_t count,
                                    int64_t total_chunks, const float* tensor_scale, int out_dtype,
                                    void* stream);

/* ---------------------------------------------------- one scale per tensor
 * [WP2] "Block scaling" ("Why not one scale for the whole matrix?") and
 * "Sixteen values aren't enough": the comparison points of block scaling.
 * Codes RN_e2m1(RN(x / scale)), one correctly rounded division per
 * element; scale = 1 rounds straight to FP4; dequantize value(code) *
 * scale.  scale must be finite and > 0 (FP4_ERR_ARG).
 *   x       [n] fp32 or bf16, 32-byte aligned; n % 16 == 0
 *   packed  [n/2] codes, 8-byte aligned
 *   y       [n] fp32 or bf16 (out_dtype), 32-byte aligned */
fp4_status fp4_scaled_quantize(const void* x, int dtype, int64_t n, float scale,
                               uint8_t* packed, void* stream);
fp4_status fp4_scaled_dequantize(const uint8_t* packed, int64_t n, float scale, void* y,
                                 int out_dtype, void* stream);

/* The same two operations with the scale in device memory, so that the one
 * scale per matrix is chosen without a round trip to the host.
 * fp4_scaled_quantize_amax: scale = RN(*amax / 6) (the largest magnitude,
 * e.g. from nvfp4_amax on x, lands on 6, the largest E2M1 value); a scale
 * that is not finite and > 0 (amax 0) is used as 1.  The scale used is
 * written to *scale_out (also for n = 0).
 *   amax, scale_out  1 fp32 each on the device, 4-byte aligned
 * fp4_scaled_dequantize_dev: value(code) * (*scale), scale a device fp32
 * (4-byte aligned) that is finite and > 0, e.g. the scale_out above.
 * Other arguments as fp4_scaled_quantize / fp4_scaled_dequantize. */
fp4_status fp4_scaled_quantize_amax(const void* x, int dtype, int64_t n, const float* amax,
                                    float* scale_out, uint8_t* packed, void* stream);
fp4_status fp4_scaled_dequantize_dev(const uint8_t* packed, int64_t n, const float* scale,
                                     void* y, int out_dtype, void* stream);

/* ------------------------------------------------------------------ MXFP4
 * [MoE-FP4] "方法概述" / "核心技术贡献" 2 (BF16ToFP4Row): each row in
 * 32-element blocks, one UE8M0 scale per block ([WP2] "Block scaling": a
 * power of two): E = floor(log2(block amax)) - 2, clamped to [-127, 127]
 * (E = -127 for an all-zero block), scale byte E + 127, codes
 * RN_e2m1(x * 2^-E) with [6, 8) saturating to 6.
 *   x       [rows, cols] fp32 or bf16 row-major, 32-byte aligned
 *   packed  [rows, cols/2] out, 16-byte aligned
 *   scales  [rows, cols/32] UE8M0 bytes out
 *   cols % 32 == 0 */
fp4_status mxfp4_quantize(const void* x, int dtype, int64_t rows, int64_t cols,
                          uint8_t* packed, uint8_t* scales, void* stream);

/* ------------------------------------------------ backward-path FP4
 * [MoE-FP4] "方法概述": gradients travel and are stored in FP8 (E4M3 with one
 * scale per 128 elements), because on Hopper the FP4 dequantize cost more
 * than the exchange saved; "局限与未来方向" names FP4 for the backward pass
 * as future work.  These two calls complete that path with
 * fp4_to_fp8_row (below): FP8 -> MXFP4 for the exchange, MXFP4 -> FP8 or
 * floats on the receiving side.
 */

/* FP8 -> MXFP4.  Each value is RN_fp32(e4m3(byte) * fp8_scales[k / 128]);
 * the values are then quantized by the mxfp4_quantize rule.
 *   fp8         [rows, cols] E4M3 bytes, 32-byte aligned (NaN bytes are
 *               outside the contract)
 *   fp8_scales  [rows, cols/128] fp32, 4-byte aligned
 *   packed      [rows, cols/2] out, 16-byte aligned
 *   scales      [rows, cols/32] UE8M0 bytes out
 *   cols % 128 == 0 */
fp4_status fp8_to_fp4_row(const uint8_t* fp8, const float* fp8_scales, int64_t rows,
                          int64_t cols, uint8_t* packed, uint8_t* scales, void* stream);

/* MXFP4 -> floats: y = value(code) * 2^(S - 127), S = 0 giving 2^-127;
 * S = 255 is the format's NaN and makes every value of its block the quiet
 * NaN 0x7FC00000 (bf16 0x7FC0).  Exact for fp32 output; bf16 output holds
 * every such value as well.
 *   packed  [rows, cols/2], 16-byte aligned; scales [rows, cols/32] UE8M0
 *   y       [rows, cols] fp32 or bf16 (out_dtype) out, 32-byte aligned
 *   cols % 32 == 0 */
fp4_status mxfp4_dequantize(const uint8_t* packed, const uint8_t* scales, int64_t rows,
                            int64_t cols, void* y, int out_dtype, void* stream);

/* ------------------------------------------------------ MXFP4 -> FP8 E4M3
 * [MoE-FP4] "核心技术贡献" 1: direct bit conversion, E_fp8 = E_fp4 - 1 + 7,
 * the mantissa bit shifted into the E4M3 mantissa field; four MXFP4 blocks
 * form one FP8 block of 128 whose scale S_t is the largest of the four UE8M0
 * scales, and each element's exponent drops by S_t - S_sub.  Defined result:
 * the E4M3 value nearest to value(code) * 2^-(S_t - S_sub) (exact unless it
 * underflows, i.e. unless S_t - S_sub >= 9); fp32 scale 2^(S_t - 127).
 */

/* FP4RowToFP8Row.
 *   packed      [rows, cols/2], 32-byte aligned; scales [rows, cols/32] UE8M0
 *   fp8         [rows, cols] E4M3 out, 32-byte aligned
 *   fp8_scales  [rows, cols/128] fp32 out, 16-byte aligned
 *   cols % 128 == 0 */
fp4_status fp4_to_fp8_row(const uint8_t* packed, const uint8_t* scales, int64_t rows,
                          int64_t cols, uint8_t* fp8, float* fp8_scales, void* stream);

/* FP4RowToFP8Col ([MoE-FP4] "核心技术贡献" 2 and 3): dequantize, transpose
 * and requantize per expert segment, over ragged segments given by
 * precomputed offsets.  Segment e holds source rows seg_row_off[e] ..
 * seg_row_off[e+1]-1 (n_e rows, n_e >= 0, non-decreasing offsets,
 * seg_row_off[0] = 0, seg_row_off[E] = total_rows) and becomes:
 *   fp8_t + cols * seg_row_off[e]:          [cols, n_e] E4M3, row-major;
 *   fp8_t_scales + cols * seg_scale_off[e]: [cols, ceil(n_e/128)] fp32,
 * where seg_scale_off is the running sum of ceil(n_e/128) (fp4_seg_scale_offsets).
 * Output row k, token block b: S_t = the largest source scale among the block's
 * (<= 128) tokens for feature block k/32.
 *   packed [total_rows, cols/2], scales [total_rows, cols/32] (as the row form)
 *   seg_row_off, seg_scale_off  device int64 [num_segments + 1]
 *   total_blocks  = seg_scale_off[num_segments] (host copy, sizes the grid),
 *                   below 2^31
 *   cols % 128 == 0.  Offsets are trusted: the device reads them as given.
 * Alignment: packed 32 bytes, scales and fp8_t_scales 4, the offsets 8;
 * fp8_t may start at any byte (the kernel stores whole 32-byte sectors and
 * writes only the partial sectors at its ends byte by byte).  FP4_ERR_ALIGN
 * otherwise; FP4_ERR_CUDA if the launch fails (it uses about 97 KB of
 * shared memory per CTA). */
fp4_status fp4_to_fp8_col(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                          const int64_t* seg_row_off, const int64_t* seg_scale_off,
                          int32_t num_segments, int64_t total_rows, int64_t total_blocks,
                          uint8_t* fp8_t, float* fp8_t_scales, void* stream);

/* FP4RowToFP8Col with the kernel's work split fixed by the caller: one CTA
 * converts a run of run_blocks consecutive 128-token blocks (in the global
 * block order of seg_scale_off) for 256 features at a time.  run_blocks = 0
 * lets the library choose (fp4_to_fp8_col does): the run length, between 8
 * and 40 blocks, whose units fill whole waves of resident CTAs.  The output
 * does not depend on it.  Errors as fp4_to_fp8_col, and FP4_ERR_SHAPE for
 * run_blocks < 0 or above 2^20. */
fp4_status fp4_to_fp8_col_runs(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                               const int64_t* seg_row_off, const int64_t* seg_scale_off,
                               int32_t num_segments, int64_t total_rows, int64_t total_blocks,
                               int32_t run_blocks, uint8_t* fp8_t, float* fp8_t_scales,
                               void* stream);

/* Host helper: host_scale_off[0] = 0, host_scale_off[e+1] = host_scale_off[e]
 * + ceil((host_row_off[e+1] - host_row_off[e]) / 128).  Returns FP4_ERR_SHAPE
 * on a decreasing offset. */
fp4_status fp4_seg_scale_offsets(const int64_t* host_row_off, int32_t num_segments,
                                 int64_t* host_scale_off);

/* --------------------------------------------------------------- FP4Quant
 * [FP4Quant] "Why four bits need more than rounding": per contiguous group of
 * G in {64, 128, 256} along each row: s1 = RMS of the group (balanced
 * pairwise sum of squares), y = x * RN(1/s1), z = normalized Walsh-Hadamard
 * transform of y (butterflies h = 1, 2, ..., G/2, then times RN(1/sqrt(G))),
 * s2 = max|z| / 6, codes = RN_e2m1(z * RN(1/s2)); both scales are stored.
 * "Making compression cheap enough to help": the decode unpacks,
 * dequantizes (z' = value * s2), runs the inverse transform (the same
 * normalized transform) and undoes the RMS scale (x' = y' * s1).
 *   x / y   [rows, cols] fp32 or bf16, 32-byte aligned
 *   packed  [rows, cols/2], 16-byte aligned
 *   s1, s2  [rows, cols/G] fp32, 4-byte aligned
 *   cols % G == 0
 * Errors: FP4_ERR_SHAPE for negative sizes, cols % G != 0 or rows * cols
 * above 2^40 elements. */
fp4_status fp4quant_encode(const void* x, int dtype, int64_t rows, int64_t cols, int group,
                           uint8_t* packed, float* s1, float* s2, void* stream);
fp4_status fp4quant_decode(const uint8_t* packed, const float* s1, const float* s2,
                           int64_t rows, int64_t cols, int group, void* y, int out_dtype,
                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4CODEC_H */
