/*
 * fp4_oracle.h -- the CPU oracle for block-scaled FP4 (E2M1) quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of what the CUDA library computes.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or constant generator with the CUDA library,
 * and neither side includes or links the other.
 *
 * Sources (cited by short key throughout):
 *   [FP4Quant]  cybernoise.de, "FP4Quant speeds up GPU communication, with a
 *               measurable accuracy trade-off" (news summary of the FP4Quant
 *               preprint).
 *   [fp4-train] huggingface.co/kernels/phanerozoic/fp4-train, model card
 *               "fp4-train".
 *   [MoE-FP4]   paper-daily.com review (2026-03-05) of "Practical FP4 Training
 *               for Large-Scale MoE Models on Hopper GPUs".
 *   [WP2]       hiren.me, "Weight precision, part 2".
 *
 * Arithmetic: every float (fp32) operation is written as its own C expression
 * and the file is compiled with -ffp-contract=off and without fast-math, so
 * each +, -, *, / and sqrtf is one IEEE-754 binary32 operation rounded to
 * nearest-even.  The pages do not fix the arithmetic precision; the quantized
 * codes are integer decisions, so the oracle takes them in the precision the
 * kernels compute in (fp32), in the operation order written below.  Format
 * encoders work from the exact value (in double where the value is exact).
 *
 * Inputs outside the contract: NaN and infinite inputs.  The oracle still
 * returns a deterministic result for them, but the parity tests never feed
 * them.
 */
#ifndef FP4_ORACLE_H
#define FP4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- formats */

/* Value of a 4-bit E2M1 code: bit 3 sign, bits 2:1 exponent, bit 0 mantissa.
 * [WP2] "What FP4 can hold" (grid table). */
double ora_e2m1_value(uint8_t code);

/* Round-to-nearest E2M1 encode of a float: nearest grid value, ties to the
 * code whose mantissa bit is 0, |a| >= 6 saturates to 6, the sign bit is
 * copied from the input (so -0.1 -> code 0x8).  [WP2] "Sixteen values aren't
 * enough" (values below 0.25 round to 0); [fp4-train] "How it works". */
uint8_t ora_e2m1_rn(float a);

/* Stochastic E2M1 encode: between grid neighbours lo <= |a| < hi the upper one
 * is taken when u < (|a| - lo) / (hi - lo), u = (word >> 8) * 2^-24.
 * [fp4-train] "How it works". */
uint8_t ora_e2m1_sr(float a, uint32_t word);

/* OCP E4M3FN: bias 7, largest finite 448, subnormal step 2^-9, no infinity.
 * Encode rounds the exact value to nearest-even and saturates to +-448. */
double ora_e4m3_value(uint8_t b);
uint8_t ora_e4m3_rn_d(double x);
uint8_t ora_e4m3_rn(float x);

/* UE8M0 (MX shared scale): value 2^(b-127). */
double ora_ue8m0_value(uint8_t b);

/* bfloat16 <-> float; float -> bf16 rounds to nearest-even, NaN stays NaN. */
uint16_t ora_bf16_rn(float x);
float ora_bf16_value(uint16_t b);

/* ----------------------------------------------------------------- Philox */

/* Philox4x32 with 10 rounds, from Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3" (SC'11). */
void ora_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The random word for flat element index g of a tensor quantized at (seed,
 * step): a 16-bit uniform h, returned as h << 16 so that the stochastic rule's
 * u = (word >> 8) * 2^-24 is h * 2^-16.  h is half g & 1 (low half first) of
 * word (g >> 1) & 3 of Philox4x32-10 at counter (g>>3 lo, g>>3 hi, step lo,
 * step hi), key (seed lo, seed hi): one call serves eight elements.
 * [fp4-train] "How it works" (counter-based RNG keyed on seed, step and
 * global index; the upper neighbour taken with probability equal to the
 * fractional distance, here to within 2^-16). */
uint32_t ora_rng_word(uint64_t seed, uint64_t step, uint64_t g);

/* ------------------------------------------------------------------ NVFP4 */

enum { ORA_RTN = 0, ORA_SR = 1 };
enum { ORA_TSCALE_GIVEN = 0, ORA_TSCALE_COMPUTE = 1 };

/* max |x[i] (+ r[i])| over n elements (r may be NULL); NaN ignored. */
float ora_nvfp4_amax(const float* x, const float* r, int64_t n);

/* Per-tensor scale from the tensor amax: amax / (6 * 448); a result that is
 * not finite or not > 0 is replaced by 1.  [WP2] "Block scaling" (one 32-bit
 * scale for the whole matrix). */
float ora_nvfp4_tensor_scale(float amax);

/* A caller-given tensor scale that is not finite or not > 0 is used as 1. */
float ora_nvfp4_sanitize_scale(float s);

/* One 16-element block v[0..15] (already including any residual) with tensor
 * scale s_t.  Writes 8 packed bytes (element 2i in the low nibble), the e4m3
 * block scale and the dequantized fp32 values q[16].  g0 is the flat index of
 * v[0], used only by stochastic rounding.  [fp4-train] "How it works". */
void ora_nvfp4_block(const float v[16], float s_t, int rounding, uint64_t seed,
                     uint64_t step, uint64_t g0, uint8_t packed[8],
                     uint8_t* scale, float q[16]);

/* Whole-tensor quantize of n floats (n % 16 == 0).  residual (nullable) is
 * read and updated in place (error feedback).  tensor_scale: read in GIVEN
 * mode, written in COMPUTE mode.  Returns 0, or -1 on a bad argument. */
int ora_nvfp4_quantize(const float* x, int64_t n, float* residual, int rounding,
                       uint64_t seed, uint64_t step, int tscale_mode,
                       float* tensor_scale, uint8_t* packed, uint8_t* scales);

/* y[i] = value(code_i) * (e4m3(scale_b) * s_t), one fp32 product each. */
int ora_nvfp4_dequantize(const uint8_t* packed, const uint8_t* scales,
                         float tensor_scale, int64_t n, float* y);

/* The fused update-quantize-dequantize of one training step on a bf16 weight:
 * v = ((W - lr*G) + r); quantize v; W <- bf16(q); r <- v - q.  g and residual
 * may be NULL.  [fp4-train] "Usage" (ErrorFeedback.qdq of W - lr*grad). */
int ora_nvfp4_qdq(uint16_t* w, const float* g, float lr, int64_t n,
                  float* residual, int rounding, uint64_t seed, uint64_t step,
                  int tscale_mode, float* tensor_scale, uint8_t* packed,
                  uint8_t* scales);

/* max |v| of the qdq update v = (W - lr*G) + r, for the COMPUTE scale. */
float ora_nvfp4_qdq_amax(const uint16_t* w, const float* g, float lr,
                         const float* residual, int64_t n);

/* ------------------------------------------------------------------ MXFP4 */

/* One row of cols floats (cols % 32 == 0): per 32-block a UE8M0 scale byte
 * floor(log2 max|x|) - 2 + 127 (clamped to [0, 254]; 0 for an all-zero
 * block) and codes RN_e2m1(x * 2^-E).  [MoE-FP4] "方法概述" (MXFP4: E2M1,
 * 32-element blocks, UE8M0 scale); [WP2] "Block scaling" (power-of-two
 * scale). */
/* One fp32 scale per tensor ([WP2] "Block scaling", "Sixteen values aren't
 * enough"): codes RN_e2m1(RN(x / s)); s = 1 rounds straight to FP4. */
int ora_fp4_scaled_quantize(const float* x, int64_t n, float s, uint8_t* packed);
int ora_fp4_scaled_dequantize(const uint8_t* packed, int64_t n, float s, float* y);

int ora_mxfp4_quantize_row(const float* x, int64_t cols, uint8_t* packed,
                           uint8_t* scales);

/* ------------------------------------------------------- MXFP4 -> FP8 E4M3 */

/* Row form, one row (cols % 128 == 0): per 128-span the target scale is the
 * largest of its four UE8M0 bytes S_t, the fp32 output scale is 2^(S_t-127)
 * and each element becomes RN_e4m3(value(code) * 2^-(S_t - S_sub)).
 * [MoE-FP4] "核心技术贡献" 1 (direct FP4-to-FP8 bit conversion, hierarchical
 * scale alignment). */
/* Backward-path FP4: E4M3 values times their per-128 fp32 scale, rounded
 * to fp32, quantized to MXFP4 ([MoE-FP4] "局限与未来方向"). */
int ora_fp8_to_fp4_row(const uint8_t* fp8, const float* fp8_scales, int64_t cols,
                       uint8_t* packed, uint8_t* scales);
int ora_fp8_to_fp4_rows(const uint8_t* fp8, const float* fp8_scales, int64_t rows,
                        int64_t cols, uint8_t* packed, uint8_t* scales);
int ora_mxfp4_dequantize(const uint8_t* packed, const uint8_t* scales, int64_t rows,
                         int64_t cols, float* y);
/* MXFP4 -> fp32: value(code) * 2^(S - 127). */
int ora_mxfp4_dequantize_row(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                             float* y);
int ora_fp4_to_fp8_row(const uint8_t* packed, const uint8_t* scales,
                       int64_t cols, uint8_t* fp8, float* fp8_scales);

/* Column form for one expert segment: rows row0 .. row0+n_e-1 of the packed
 * [*, cols] tensor become the row-major [cols, n_e] E4M3 matrix out and the
 * [cols, ceil(n_e/128)] fp32 scales out_scales.  Each element is dequantized
 * exactly, transposed, and requantized against 2^(S_t-127), S_t the largest
 * source scale among the <= 128 tokens of its output block.  [MoE-FP4]
 * "核心技术贡献" 2 (FP4RowToFP8Col) and 3 (ragged segments). */
int ora_fp4_to_fp8_col_segment(const uint8_t* packed, const uint8_t* scales,
                               int64_t cols, int64_t row0, int64_t n_e,
                               uint8_t* out, float* out_scales);

/* ------------------------------------------------------ blocked scale layout */

/* Bytes of the blocked form of a [rows, cols] one-byte scale matrix:
 * 128 * ceil(rows / 128) * 4 * ceil(cols / 4); -1 for negative sizes. */
int64_t ora_blocked_scales_size(int64_t rows, int64_t cols);

/* [rows, cols] row-major scales -> the blocked layout that block-scaled
 * tensor-core matmuls read: zero padding to whole 128 x 4 tiles, tiles in
 * row-major order, the scale of tile row r, column c at byte
 * 16 * (r % 32) + 4 * (r / 32) + c of its 512-byte tile.  [fp4-train]
 * "Scope" (scales swizzled for torch._scaled_mm); the layout itself follows
 * the public description of the tensor cores' block-scale layout. */
int ora_scales_to_blocked(const uint8_t* scales, int64_t rows, int64_t cols,
                          uint8_t* blocked);

/* The inverse: the [rows, cols] scales read back out of the blocked form. */
int ora_scales_from_blocked(const uint8_t* blocked, int64_t rows, int64_t cols,
                            uint8_t* scales);

/* ------------------------------------------------------------------ FP4Quant */

/* The normalization constant RN(1/sqrt(G)) for G in {64, 128, 256}. */
float ora_wht_norm(int group);

/* In-place normalized Walsh-Hadamard transform of G floats: butterflies
 * (a, b) -> (a + b, a - b) for h = 1, 2, ..., G/2, then every element times
 * RN(1/sqrt(G)).  [FP4Quant] "Why four bits need more than rounding". */
void ora_wht(float* y, int group);

/* One row (cols % G == 0): per group an RMS scale s1, the normalized WHT of
 * x / s1, an absmax scale s2 = max|z| / 6 and E2M1 codes of z / s2.
 * [FP4Quant] "Why four bits need more than rounding", "Making compression
 * cheap enough to help". */
int ora_fp4quant_encode_row(const float* x, int64_t cols, int group,
                            uint8_t* packed, float* s1, float* s2);

/* The inverse: z = value * s2, y = WHT(z), x = y * s1. */
int ora_fp4quant_decode_row(const uint8_t* packed, const float* s1,
                            const float* s2, int64_t cols, int group, float* x);

#ifdef __cplusplus
}
#endif

#endif /* FP4_ORACLE_H */
