/*
 * fp4quant.c -- oracle: FP4Quant group encode / decode.  Test infrastructure
 * only (see fp4_oracle.h).
 *
 * [FP4Quant] "Why four bits need more than rounding": the tensor is split
 * into small contiguous groups; each group first gets a scale from its
 * root-mean-square magnitude, then a normalized Walsh-Hadamard transform made
 * of additions and subtractions, then a second scale from the largest
 * absolute transformed value that fits the group into the FP4 range; both
 * scales travel with the codes.  "Making compression cheap enough to help":
 * the receiver unpacks, dequantizes and runs the inverse transform.
 *
 * Where the page leaves the order open: the sum of squares is a balanced
 * pairwise tree over adjacent elements; a scale is applied by multiplying by
 * its correctly rounded reciprocal (0 for a zero scale); the transform runs
 * its butterfly stages h = 1, 2, 4, ... in natural (Sylvester) order and then
 * multiplies by RN(1/sqrt(G)); the normalized transform is its own inverse.
 */
#include "fp4_oracle.h"

#include <math.h>

float ora_wht_norm(int group) {
  if (group == 64) return 0.125f;
  if (group == 256) return 0.0625f;
  if (group == 128) return sqrtf(2.0f) * 0.0625f; /* 2^-3.5 = sqrt(2) / 16 */
  return 0.0f;
}

void ora_wht(float* y, int group) {
  for (int h = 1; h < group; h *= 2) {
    for (int i = 0; i < group; ++i) {
      if (i & h) continue;
      float a = y[i];
      float b = y[i + h];
      y[i] = a + b;
      y[i + h] = a - b;
    }
  }
  float c = ora_wht_norm(group);
  for (int i = 0; i < group; ++i) y[i] = y[i] * c;
}

static int group_ok(int g) { return g == 64 || g == 128 || g == 256; }

int ora_fp4quant_encode_row(const float* x, int64_t cols, int group,
                            uint8_t* packed, float* s1, float* s2) {
  if (!group_ok(group) || cols < 0 || cols % group != 0) return -1;
  for (int64_t gi = 0; gi < cols / group; ++gi) {
    const float* xg = x + gi * group;
    float sq[256], y[256];
    /* RMS: balanced pairwise sum of squares over adjacent pairs. */
    for (int i = 0; i < group; ++i) sq[i] = xg[i] * xg[i];
    for (int width = group; width > 1; width /= 2)
      for (int i = 0; i < width / 2; ++i) sq[i] = sq[2 * i] + sq[2 * i + 1];
    float mean_sq = sq[0] * (1.0f / (float)group);
    float rms = sqrtf(mean_sq);
    float inv1 = (rms == 0.0f) ? 0.0f : 1.0f / rms;
    for (int i = 0; i < group; ++i) y[i] = xg[i] * inv1;
    /* Normalized Walsh-Hadamard transform. */
    ora_wht(y, group);
    /* Absmax scale into the E2M1 range (largest value 6). */
    float zmax = 0.0f;
    for (int i = 0; i < group; ++i) zmax = fmaxf(zmax, fabsf(y[i]));
    float sc2 = zmax / 6.0f;
    float inv2 = (sc2 == 0.0f) ? 0.0f : 1.0f / sc2;
    for (int i = 0; i < group; i += 2) {
      uint8_t c0 = ora_e2m1_rn(y[i] * inv2);
      uint8_t c1 = ora_e2m1_rn(y[i + 1] * inv2);
      packed[(gi * group + i) / 2] = (uint8_t)(c0 | (c1 << 4));
    }
    s1[gi] = rms;
    s2[gi] = sc2;
  }
  return 0;
}

int ora_fp4quant_decode_row(const uint8_t* packed, const float* s1,
                            const float* s2, int64_t cols, int group, float* x) {
  if (!group_ok(group) || cols < 0 || cols % group != 0) return -1;
  for (int64_t gi = 0; gi < cols / group; ++gi) {
    float z[256];
    for (int i = 0; i < group; ++i) {
      int64_t k = gi * group + i;
      uint8_t byte = packed[k / 2];
      uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
      z[i] = (float)ora_e2m1_value(code) * s2[gi];
    }
    ora_wht(z, group);
    for (int i = 0; i < group; ++i) x[gi * group + i] = z[i] * s1[gi];
  }
  return 0;
}
