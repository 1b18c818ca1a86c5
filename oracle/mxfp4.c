/*
 * mxfp4.c -- oracle: MXFP4 quantize and the direct MXFP4 -> FP8 E4M3
 * conversions.  Test infrastructure only (see fp4_oracle.h).
 */
#include "fp4_oracle.h"

#include <math.h>

/* [MoE-FP4] "方法概述": activations become MXFP4, E2M1 elements with one
 * UE8M0 scale per 32 elements.  [WP2] "Block scaling": that scale is a power
 * of two.  The exponent is the one of the OCP microscaling rule the fp4-train
 * card refers to: floor(log2(block amax)) minus 2, the exponent of the
 * largest E2M1 value, so the block amax lands in [4, 8) and values from 6 up
 * saturate to 6. */
int ora_mxfp4_quantize_row(const float* x, int64_t cols, uint8_t* packed,
                           uint8_t* scales) {
  if (cols < 0 || cols % 32 != 0) return -1;
  for (int64_t b = 0; b < cols / 32; ++b) {
    const float* xb = x + 32 * b;
    float bmax = 0.0f;
    for (int i = 0; i < 32; ++i) bmax = fmaxf(bmax, fabsf(xb[i]));
    int E;
    if (bmax == 0.0f) {
      E = -127;
    } else if (isinf(bmax)) {
      /* the exponent field of an infinite amax is 255: floor(log2) read
       * from it is 128 (frexpf leaves the exponent of an infinity
       * unspecified); the infinite elements then saturate to +-6 */
      E = 128 - 2;
    } else {
      int e2;
      frexpf(bmax, &e2);       /* bmax = f * 2^e2, f in [0.5, 1) */
      E = (e2 - 1) - 2;        /* floor(log2 bmax) - emax(E2M1) */
      if (E < -127) E = -127;
      if (E > 127) E = 127;
    }
    scales[b] = (uint8_t)(E + 127);
    for (int i = 0; i < 32; i += 2) {
      uint8_t c0 = ora_e2m1_rn(ldexpf(xb[i], -E));
      uint8_t c1 = ora_e2m1_rn(ldexpf(xb[i + 1], -E));
      packed[16 * b + i / 2] = (uint8_t)(c0 | (c1 << 4));
    }
  }
  return 0;
}

static uint8_t code_at(const uint8_t* packed_row, int64_t k) {
  uint8_t byte = packed_row[k / 2];
  return (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
}

/* [MoE-FP4] "核心技术贡献" 1: four MXFP4 blocks (4 x 32) form one FP8 block
 * of 128; the largest of the four source scales is the target scale and each
 * element's exponent drops by (S_target - S_sub).  The defined result is the
 * E4M3 value nearest to value(code) * 2^-(S_t - S_sub), exact while no
 * underflow occurs. */
int ora_fp4_to_fp8_row(const uint8_t* packed, const uint8_t* scales,
                       int64_t cols, uint8_t* fp8, float* fp8_scales) {
  if (cols < 0 || cols % 128 != 0) return -1;
  for (int64_t j = 0; j < cols / 128; ++j) {
    int st = 0;
    for (int s = 0; s < 4; ++s)
      if (scales[4 * j + s] > st) st = scales[4 * j + s];
    fp8_scales[j] = ldexpf(1.0f, st - 127);
    for (int64_t k = 128 * j; k < 128 * j + 128; ++k) {
      int d = st - scales[k / 32];
      double v = ora_e2m1_value(code_at(packed, k)) * ldexp(1.0, -d);
      fp8[k] = ora_e4m3_rn_d(v);
    }
  }
  return 0;
}

/* [MoE-FP4] "核心技术贡献" 2 and 3: FP4RowToFP8Col dequantizes, transposes
 * and requantizes; expert segments are ragged and located by precomputed
 * offsets.  Written here in that order: the exact dequantized value of the
 * source element, placed at its transposed position, requantized against the
 * power-of-two scale 2^(S_t - 127) of its output block of <= 128 tokens. */
int ora_fp4_to_fp8_col_segment(const uint8_t* packed, const uint8_t* scales,
                               int64_t cols, int64_t row0, int64_t n_e,
                               uint8_t* out, float* out_scales) {
  if (cols < 0 || cols % 128 != 0 || n_e < 0 || row0 < 0) return -1;
  int64_t nb = (n_e + 127) / 128;
  int64_t spr = cols / 32; /* scale bytes per source row */
  for (int64_t k = 0; k < cols; ++k) {
    for (int64_t b = 0; b < nb; ++b) {
      int64_t j_end = (128 * b + 128 < n_e) ? 128 * b + 128 : n_e;
      int st = 0;
      for (int64_t j = 128 * b; j < j_end; ++j) {
        int s = scales[(row0 + j) * spr + k / 32];
        if (s > st) st = s;
      }
      out_scales[k * nb + b] = ldexpf(1.0f, st - 127);
      double target = ldexp(1.0, st - 127);
      for (int64_t j = 128 * b; j < j_end; ++j) {
        const uint8_t* prow = packed + (row0 + j) * (cols / 2);
        int s = scales[(row0 + j) * spr + k / 32];
        double value = ora_e2m1_value(code_at(prow, k)) * ldexp(1.0, s - 127);
        out[k * n_e + j] = ora_e4m3_rn_d(value / target);
      }
    }
  }
  return 0;
}

/* Backward-path FP4, which [MoE-FP4] "局限与未来方向" names as future work:
 * FP8 gradients ("方法概述": E4M3 with one scale per 128 elements) become
 * MXFP4 for communication.  Each element's value is the E4M3 value times its
 * block's fp32 scale, rounded once to fp32; the MXFP4 rule above then
 * quantizes those values. */
int ora_fp8_to_fp4_row(const uint8_t* fp8, const float* fp8_scales, int64_t cols,
                       uint8_t* packed, uint8_t* scales) {
  if (cols < 0 || cols % 128 != 0) return -1;
  float v[32];
  for (int64_t b = 0; b < cols / 32; ++b) {
    const double s = (double)fp8_scales[(32 * b) / 128];
    for (int i = 0; i < 32; ++i) v[i] = (float)(ora_e4m3_value(fp8[32 * b + i]) * s);
    if (ora_mxfp4_quantize_row(v, 32, packed + 16 * b, scales + b) != 0) return -1;
  }
  return 0;
}

/* MXFP4 dequantize: value(code) * 2^(S - 127) for the element's UE8M0 scale
 * S (the product of a 2-bit E2M1 value and a power of two, exact in fp32
 * unless it leaves the fp32 range). */
int ora_mxfp4_dequantize_row(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                             float* y) {
  if (cols < 0 || cols % 32 != 0) return -1;
  for (int64_t k = 0; k < cols; ++k)
    y[k] = (float)(ora_e2m1_value(code_at(packed, k)) * ora_ue8m0_value(scales[k / 32]));
  return 0;
}
