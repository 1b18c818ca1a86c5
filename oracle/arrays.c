/*
 * arrays.c -- oracle: loops over arrays and matrices of the scalar and row
 * functions, so the Python tests can call the oracle on whole tensors.  Test
 * infrastructure only (see fp4_oracle.h).
 */
#include "fp4_oracle.h"

void ora_e2m1_rn_array(const float* a, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ora_e2m1_rn(a[i]);
}

void ora_e2m1_sr_array(const float* a, const uint32_t* words, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ora_e2m1_sr(a[i], words[i]);
}

void ora_e4m3_rn_array(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ora_e4m3_rn_d(x[i]);
}

void ora_bf16_rn_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ora_bf16_rn(x[i]);
}

void ora_rng_word_array(uint64_t seed, uint64_t step, const uint64_t* g, int64_t n,
                        uint32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ora_rng_word(seed, step, g[i]);
}

/* Quantize the blocks [b0, b0 + nb) of a tensor whose block b starts at flat
 * index 16 * b, with a known tensor scale: the sampled form of
 * ora_nvfp4_quantize used on tensors too large for the whole-tensor call.
 * v holds the 16 * nb block inputs (residual already added). */
void ora_nvfp4_blocks(const float* v, int64_t b0, int64_t nb, float s_t, int rounding,
                      uint64_t seed, uint64_t step, uint8_t* packed, uint8_t* scales,
                      float* q) {
  for (int64_t b = 0; b < nb; ++b)
    ora_nvfp4_block(v + 16 * b, s_t, rounding, seed, step, (uint64_t)(16 * (b0 + b)),
                    packed + 8 * b, scales + b, q + 16 * b);
}

int ora_mxfp4_quantize(const float* x, int64_t rows, int64_t cols, uint8_t* packed,
                       uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    int rc = ora_mxfp4_quantize_row(x + r * cols, cols, packed + r * (cols / 2),
                                    scales + r * (cols / 32));
    if (rc) return rc;
  }
  return 0;
}

int ora_fp4_to_fp8_rows(const uint8_t* packed, const uint8_t* scales, int64_t rows,
                        int64_t cols, uint8_t* fp8, float* fp8_scales) {
  for (int64_t r = 0; r < rows; ++r) {
    int rc = ora_fp4_to_fp8_row(packed + r * (cols / 2), scales + r * (cols / 32), cols,
                                fp8 + r * cols, fp8_scales + r * (cols / 128));
    if (rc) return rc;
  }
  return 0;
}

int ora_fp8_to_fp4_rows(const uint8_t* fp8, const float* fp8_scales, int64_t rows,
                        int64_t cols, uint8_t* packed, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    int rc = ora_fp8_to_fp4_row(fp8 + r * cols, fp8_scales + r * (cols / 128), cols,
                                packed + r * (cols / 2), scales + r * (cols / 32));
    if (rc) return rc;
  }
  return 0;
}

int ora_mxfp4_dequantize(const uint8_t* packed, const uint8_t* scales, int64_t rows,
                         int64_t cols, float* y) {
  for (int64_t r = 0; r < rows; ++r) {
    int rc = ora_mxfp4_dequantize_row(packed + r * (cols / 2), scales + r * (cols / 32), cols,
                                      y + r * cols);
    if (rc) return rc;
  }
  return 0;
}

/* All segments: segment e covers rows off[e] .. off[e+1]-1; its output starts
 * at byte cols * off[e] and its scales at float cols * scale_off[e], where
 * scale_off is the running sum of ceil(n_e / 128). */
int ora_fp4_to_fp8_col(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                       const int64_t* off, int32_t num_segments, uint8_t* out,
                       float* out_scales) {
  int64_t sofs = 0;
  for (int32_t e = 0; e < num_segments; ++e) {
    int64_t n_e = off[e + 1] - off[e];
    if (n_e < 0) return -1;
    int rc = ora_fp4_to_fp8_col_segment(packed, scales, cols, off[e], n_e,
                                        out + cols * off[e], out_scales + cols * sofs);
    if (rc) return rc;
    sofs += (n_e + 127) / 128;
  }
  return 0;
}

int ora_fp4quant_encode(const float* x, int64_t rows, int64_t cols, int group,
                        uint8_t* packed, float* s1, float* s2) {
  if (group <= 0) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    int rc = ora_fp4quant_encode_row(x + r * cols, cols, group, packed + r * (cols / 2),
                                     s1 + r * (cols / group), s2 + r * (cols / group));
    if (rc) return rc;
  }
  return 0;
}

int ora_fp4quant_decode(const uint8_t* packed, const float* s1, const float* s2,
                        int64_t rows, int64_t cols, int group, float* x) {
  if (group <= 0) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    int rc = ora_fp4quant_decode_row(packed + r * (cols / 2), s1 + r * (cols / group),
                                     s2 + r * (cols / group), cols, group, x + r * cols);
    if (rc) return rc;
  }
  return 0;
}
