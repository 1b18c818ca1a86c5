/*
 * formats.c -- oracle: the element and scale formats, written from their
 * definitions.  Test infrastructure only (see fp4_oracle.h).
 */
#include "fp4_oracle.h"

#include <math.h>
#include <string.h>

/* Positive E2M1 values indexed by the 3 magnitude bits (exponent, mantissa):
 * 00 0 -> 0, 00 1 -> 0.5, 01 0 -> 1, 01 1 -> 1.5, 10 0 -> 2, 10 1 -> 3,
 * 11 0 -> 4, 11 1 -> 6.  [WP2] "What FP4 can hold". */
static const double kE2M1Grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double ora_e2m1_value(uint8_t code) {
  double m = kE2M1Grid[code & 7];
  return (code & 8) ? -m : m;
}

uint8_t ora_e2m1_rn(float a) {
  if (isnan(a)) return 0;
  uint8_t sign = signbit(a) ? 8 : 0;
  double m = fabs((double)a);
  if (m >= 6.0) return sign | 7;
  /* Nearest grid value; on a tie keep the even code (mantissa bit 0).  The
   * distance is exact in double wherever a tie is possible (m >= 0.25). */
  int best = 0;
  double best_d = m;
  for (int c = 1; c < 8; ++c) {
    double d = fabs(m - kE2M1Grid[c]);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

uint8_t ora_e2m1_sr(float a, uint32_t word) {
  if (isnan(a)) return 0;
  uint8_t sign = signbit(a) ? 8 : 0;
  float m = fabsf(a);
  if (m >= 6.0f) return sign | 7;
  /* lo = largest grid value <= m, hi = the next one. */
  int c = 0;
  while (c < 6 && (float)kE2M1Grid[c + 1] <= m) ++c;
  float lo = (float)kE2M1Grid[c];
  float hi = (float)kE2M1Grid[c + 1];
  float k = 1.0f / (hi - lo);    /* 2, 1 or 0.5: exact */
  float frac = (m - lo) * k;     /* m - lo is exact (Sterbenz), so is * k */
  float u = (float)(word >> 8) * 0x1p-24f;
  return (uint8_t)(sign | (u < frac ? c + 1 : c));
}

double ora_e4m3_value(uint8_t b) {
  int e = (b >> 3) & 0xF;
  int m = b & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return (b & 0x80) ? -v : v;
}

uint8_t ora_e4m3_rn_d(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double m = fabs(x);
  if (m >= 448.0) return sign | 0x7E;
  if (m == 0.0) return sign;
  /* Quantum of the binade of m (3 mantissa bits), never below the subnormal
   * step 2^-9; round m / quantum (exact) to the nearest integer, ties even. */
  int e2;
  frexp(m, &e2);
  int E = e2 - 1;
  if (E < -6) E = -6;
  double q = ldexp(1.0, E - 3);
  double n = nearbyint(m / q);
  double v = n * q;
  if (v > 448.0) v = 448.0;
  if (v == 0.0) return sign;
  frexp(v, &e2);
  int Ev = e2 - 1;
  if (Ev < -6) {
    int mant = (int)(v / ldexp(1.0, -9));
    return (uint8_t)(sign | mant);
  }
  int mant = (int)((v / ldexp(1.0, Ev) - 1.0) * 8.0);
  return (uint8_t)(sign | ((Ev + 7) << 3) | mant);
}

uint8_t ora_e4m3_rn(float x) { return ora_e4m3_rn_d((double)x); }

double ora_ue8m0_value(uint8_t b) {
  if (b == 0xFF) return NAN;
  return ldexp(1.0, (int)b - 127);
}

uint16_t ora_bf16_rn(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if (isnan(x)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

float ora_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
