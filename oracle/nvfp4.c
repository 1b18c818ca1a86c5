/*
 * nvfp4.c -- oracle: NVFP4 quantize / dequantize / error feedback.  Test
 * infrastructure only (see fp4_oracle.h).
 *
 * [fp4-train] "How it works": each 16-element block gets the scale
 * block_absmax / 6 encoded to e4m3; every element is divided by the decoded
 * scale and encoded to E2M1, by round-to-nearest or by stochastic rounding
 * from a (seed, step, global index) counter RNG; with error feedback the
 * residual x - dequant(quantize(x)) is added into the next quantization.
 * [WP2] "Block scaling": NVFP4 also carries one 32-bit scale per matrix; the
 * pages do not say how it is chosen, so it is amax / (6 * 448), which maps
 * the tensor's largest element to the largest e2m1 value under the largest
 * e4m3 block scale.
 */
#include "fp4_oracle.h"

#include <math.h>
#include <stddef.h>

float ora_nvfp4_amax(const float* x, const float* r, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = r ? x[i] + r[i] : x[i];
    m = fmaxf(m, fabsf(v));
  }
  return m;
}

float ora_nvfp4_sanitize_scale(float s) {
  if (!(s > 0.0f) || isinf(s)) return 1.0f;
  return s;
}

float ora_nvfp4_tensor_scale(float amax) {
  float s = amax / 2688.0f; /* 6 * 448 */
  return ora_nvfp4_sanitize_scale(s);
}

void ora_nvfp4_block(const float v[16], float s_t, int rounding, uint64_t seed,
                     uint64_t step, uint64_t g0, uint8_t packed[8],
                     uint8_t* scale, float q[16]) {
  /* Block scale: block amax over 6 (the largest e2m1 value), relative to the
   * tensor scale, encoded to e4m3. */
  float den6 = 6.0f * s_t;
  float bmax = 0.0f;
  for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
  float u = bmax / den6;
  uint8_t sb = ora_e4m3_rn(u);
  /* The decoded scale the elements are divided by. */
  float eff = (float)ora_e4m3_value(sb) * s_t;
  uint8_t codes[16];
  for (int i = 0; i < 16; ++i) {
    float a = (eff == 0.0f) ? v[i] * 0.0f : v[i] / eff;
    if (rounding == ORA_SR)
      codes[i] = ora_e2m1_sr(a, ora_rng_word(seed, step, g0 + (uint64_t)i));
    else
      codes[i] = ora_e2m1_rn(a);
    q[i] = (float)ora_e2m1_value(codes[i]) * eff;
  }
  for (int i = 0; i < 8; ++i)
    packed[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
  *scale = sb;
}

int ora_nvfp4_quantize(const float* x, int64_t n, float* residual, int rounding,
                       uint64_t seed, uint64_t step, int tscale_mode,
                       float* tensor_scale, uint8_t* packed, uint8_t* scales) {
  if (n < 0 || n % 16 != 0 || !tensor_scale) return -1;
  float s_t;
  if (tscale_mode == ORA_TSCALE_COMPUTE) {
    s_t = ora_nvfp4_tensor_scale(ora_nvfp4_amax(x, residual, n));
    *tensor_scale = s_t;
  } else {
    s_t = ora_nvfp4_sanitize_scale(*tensor_scale);
  }
  for (int64_t b = 0; b < n / 16; ++b) {
    float v[16], q[16];
    for (int i = 0; i < 16; ++i) {
      int64_t k = 16 * b + i;
      v[i] = residual ? x[k] + residual[k] : x[k];
    }
    ora_nvfp4_block(v, s_t, rounding, seed, step, (uint64_t)(16 * b), packed + 8 * b,
                    scales + b, q);
    if (residual)
      for (int i = 0; i < 16; ++i) residual[16 * b + i] = v[i] - q[i];
  }
  return 0;
}

int ora_nvfp4_dequantize(const uint8_t* packed, const uint8_t* scales,
                         float tensor_scale, int64_t n, float* y) {
  if (n < 0 || n % 16 != 0) return -1;
  float s_t = ora_nvfp4_sanitize_scale(tensor_scale);
  for (int64_t b = 0; b < n / 16; ++b) {
    /* [WP2] "Block scaling", step 5: multiply back by the scale. */
    float eff = (float)ora_e4m3_value(scales[b]) * s_t;
    for (int i = 0; i < 16; ++i) {
      int64_t k = 16 * b + i;
      uint8_t byte = packed[k / 2];
      uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
      y[k] = (float)ora_e2m1_value(code) * eff;
    }
  }
  return 0;
}

/* v = ((W - lr*G) + r), each step one fp32 operation. */
static float qdq_update(const uint16_t* w, const float* g, float lr,
                        const float* r, int64_t k) {
  float v = ora_bf16_value(w[k]);
  if (g) {
    float step = lr * g[k];
    v = v - step;
  }
  if (r) v = v + r[k];
  return v;
}

float ora_nvfp4_qdq_amax(const uint16_t* w, const float* g, float lr,
                         const float* residual, int64_t n) {
  float m = 0.0f;
  for (int64_t k = 0; k < n; ++k) m = fmaxf(m, fabsf(qdq_update(w, g, lr, residual, k)));
  return m;
}

int ora_nvfp4_qdq(uint16_t* w, const float* g, float lr, int64_t n,
                  float* residual, int rounding, uint64_t seed, uint64_t step,
                  int tscale_mode, float* tensor_scale, uint8_t* packed,
                  uint8_t* scales) {
  if (n < 0 || n % 16 != 0 || !tensor_scale) return -1;
  float s_t;
  if (tscale_mode == ORA_TSCALE_COMPUTE) {
    s_t = ora_nvfp4_tensor_scale(ora_nvfp4_qdq_amax(w, g, lr, residual, n));
    *tensor_scale = s_t;
  } else {
    s_t = ora_nvfp4_sanitize_scale(*tensor_scale);
  }
  for (int64_t b = 0; b < n / 16; ++b) {
    float v[16], q[16];
    for (int i = 0; i < 16; ++i) v[i] = qdq_update(w, g, lr, residual, 16 * b + i);
    ora_nvfp4_block(v, s_t, rounding, seed, step, (uint64_t)(16 * b), packed + 8 * b,
                    scales + b, q);
    for (int i = 0; i < 16; ++i) {
      int64_t k = 16 * b + i;
      w[k] = ora_bf16_rn(q[i]);
      if (residual) residual[k] = v[i] - q[i];
    }
  }
  return 0;
}

/* [WP2] "Block scaling" ("Why not one scale for the whole matrix?") and
 * "Sixteen values aren't enough" (rounding straight to FP4): one fp32 scale
 * s for the whole tensor, each code RN_e2m1(RN(x / s)), the division being
 * one correctly rounded fp32 operation as in the block rule; s = 1 is
 * rounding straight to FP4.  The quality comparison of that page's table
 * uses both. */
int ora_fp4_scaled_quantize(const float* x, int64_t n, float s, uint8_t* packed) {
  if (n < 0 || n % 2 != 0 || !(s > 0.0f) || isinf(s)) return -1;
  for (int64_t i = 0; i < n; i += 2) {
    const float a = x[i] / s, b = x[i + 1] / s;
    packed[i / 2] = (uint8_t)(ora_e2m1_rn(a) | (ora_e2m1_rn(b) << 4));
  }
  return 0;
}

int ora_fp4_scaled_dequantize(const uint8_t* packed, int64_t n, float s, float* y) {
  if (n < 0 || n % 2 != 0) return -1;
  for (int64_t i = 0; i < n; ++i) {
    const uint8_t c = (i & 1) ? (uint8_t)(packed[i / 2] >> 4) : (uint8_t)(packed[i / 2] & 0xF);
    y[i] = (float)ora_e2m1_value(c) * s;
  }
  return 0;
}
