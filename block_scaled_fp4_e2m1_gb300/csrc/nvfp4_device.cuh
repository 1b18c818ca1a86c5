// nvfp4_device.cuh -- device code shared by the NVFP4 kernels of nvfp4.cu
// (one tensor per launch) and nvfp4_batched.cu (a list of tensors per
// launch): scale arithmetic, block loads and stores, the quantization of one
// 16-element block and the decode of 16 codes.
//
// [fp4-train] "How it works": 16-element blocks, scale block_absmax / 6
// encoded to e4m3, every element divided by the decoded scale and encoded to
// E2M1 by round-to-nearest or by stochastic rounding from a counter-based
// (seed, step, global index) RNG.  [WP2] "Block scaling": one fp32 scale per
// tensor besides the block scales (chosen as amax / (6 * 448)).
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "rn_math.cuh"

namespace fp4 {
namespace {


constexpr int kThreads = 256;

// A tensor scale that is not finite or not > 0 is used as 1.
__device__ __forceinline__ float sanitize_scale(float s) {
  return (s > 0.0f && s <= 3.40282347e38f) ? s : 1.0f;
}

__device__ __forceinline__ float tensor_scale_from_amax(float amax) {
  return sanitize_scale(__fdiv_rn(amax, 2688.0f));  // 6 * 448
}

__device__ __forceinline__ void load_f32x16(const float* p, float v[16]) {
  U32x8 a = ld_v8(p), c = ld_v8(p + 8);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = __uint_as_float(a.w[i]);
    v[8 + i] = __uint_as_float(c.w[i]);
  }
}

__device__ __forceinline__ void load_f32x16_stream(const float* p, float v[16]) {
  U32x8 a = ld_stream_v8(p), c = ld_stream_v8(p + 8);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = __uint_as_float(a.w[i]);
    v[8 + i] = __uint_as_float(c.w[i]);
  }
}

__device__ __forceinline__ void store_f32x16(float* p, const float v[16]) {
  U32x8 a, c;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a.w[i] = __float_as_uint(v[i]);
    c.w[i] = __float_as_uint(v[8 + i]);
  }
  st_v8(p, a);
  st_v8(p + 8, c);
}

// Block-level max of non-negative floats into *out (atomic, order-free).
__device__ __forceinline__ void block_max_to(float m, float* out) {
  __shared__ uint32_t warp_max[kThreads / 32];
  uint32_t u = warp_max_u32(__float_as_uint(m));
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_max[warp] = u;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kThreads / 32 ? warp_max[lane] : 0u;
    w = warp_max_u32(w);
    if (lane == 0 && w != 0u) atomicMax(reinterpret_cast<unsigned int*>(out), w);
  }
}

// Exact ties of bf16 quotients.  Let the dividend have at most 8
// significant bits (a bf16 value) and the divisor y = m * 2^k, m odd, have
// m < 2^14 (the low 10 bits of its significand are zero: "short").  Every
// rounding midpoint M of E2M1 or E4M3 is j * 2^s with j odd, j < 32.  If
// x / y != M, then |x - M*y| is a nonzero multiple of the coarser of the two
// quanta of x and M*y, which puts x / y at a relative distance of at least
// min(1 / (j*m), 2^-8) > 2^-19 from M.  The bracket (below) spans less than
// 2^-20 relative, so when its two codes differ, x / y == M exactly:
// RN(x / y) is the midpoint itself, and the code is the even one of the two.
// Divisors of this kind are common: the tensor scale amax / (6 * 448)
// carries the factors 3 and 7, which bf16 maxima often cancel.
__device__ __forceinline__ bool short_divisor(float y) {
  return (__float_as_uint(y) & 0x3FFu) == 0u;
}

// Per-kernel constants of the block-scale division u = bmax / den6.
struct ScaleDiv {
  float den6;    // 6 * s_t
  float r_lo;    // RN(RN(1/den6) * (1 - 2^-21)), 0 when den6 is outside [2^-125, 2^125]
  float r_hi;    // RN(RN(1/den6) * (1 + 2^-21))
  bool short6;   // den6 certified and short (see short_divisor)
};

__device__ __forceinline__ ScaleDiv make_scale_div(float s_t) {
  ScaleDiv d;
  d.den6 = __fmul_rn(6.0f, s_t);
  if (d.den6 >= 0x1p-125f && d.den6 <= 0x1p125f) {
    const float r = __frcp_rn(d.den6);
    d.r_lo = __fmul_rn(r, 0x1.fffffp-1f);
    d.r_hi = __fmul_rn(r, 0x1.000008p+0f);
  } else {
    d.r_lo = d.r_hi = 0.0f;
  }
  d.short6 = d.r_lo != 0.0f && short_divisor(d.den6);
  return d;
}

// Certified rounding without a division.  For q = RN(x / y) and an encoder
// E that is monotone in its argument (RN_e4m3, RN_e2m1: both keep the sign,
// round to nearest and saturate), let r = RN(1/y) with y a normal float in
// [2^-125, 2^125], L = RN(x * RN(r * (1 - 2^-21))) and
// H = RN(x * RN(r * (1 + 2^-21))).  Each of the three roundings has relative
// error <= 2^-24, so (1 - 2^-21)(1 + 2^-24)^3 < 1 - 2^-24 and
// (1 + 2^-21)(1 - 2^-24)^3 > 1 + 2^-24 put q between L and H whenever x / y
// is a normal float (below that all three are far under the smallest
// nonzero E2M1 or E4M3 magnitude and encode to the same signed zero; above
// it all saturate).  Hence E(L) == E(H) implies E(q) == E(L); otherwise the
// caller divides exactly.

// Exact fallbacks of the certified fast paths, kept out of line so that the
// compiler cannot evaluate them speculatively on the common path.
__device__ __noinline__ uint32_t exact_e4m3_quotient(float x, float y) {
  return cvt_e4m3(__fdiv_rn(x, y));
}

__device__ __noinline__ uint32_t exact_e2m1_quotient(float x, float y) {
  return cvt_e2m1x2(__fdiv_rn(x, y), 0.0f) & 0xFu;
}

// The stochastic-rounding code of RN(x / y) by the rule of e2m1_sr, with an
// exact division (the fallback of sr_codes8).
__device__ __noinline__ uint32_t exact_e2m1_sr_quotient(float x, float y, uint32_t rw) {
  return e2m1_sr(y == 0.0f ? __fmul_rn(x, 0.0f) : __fdiv_rn(x, y), rw);
}

// Stochastic rounding without a division.  For m = |a| < 6 the code of
// e2m1_sr is c + [u < frac], c the grid interval of m and frac its position
// in it; with the position s = c + frac that is ceil(s - u) (u < 1), and
// s(m) is piecewise linear and continuous: 2m below 2, m + 2 on [2, 4),
// m/2 + 4 on [4, 6), and 7 from 6 on (code 7), which is
// min(2m, m + 2, m/2 + 4, 7).  Here a = RN(x / eff) is replaced by
// q = RN(x * inv), inv = RN(1/eff) with eff in [2^-125, 2^125]:
// |q - a| <= 1.5 * 2^-23 |x / eff|, and with slopes <= 2 the position moves
// by at most 1.5 * 2^-21.  The code is taken as RN(T) with
// T = RN(min(2m + 1/2, m + 5/2, m/2 + 9/2, 15/2) - u) ~ ceil(s - u) + ...:
// ceil(t) = RN(t + 1/2) for non-integer t.  The roundings of the pieces and
// of the difference add at most 2^-21 + 2^-22, so T is within 2^-19 of
// t + 1/2, t = s(a) - u; when T lies more than 2^-19 inside its rounding
// interval, RN(T) is a's code.  Otherwise (about one element in 10^5, and
// NaN) the element's group of eight is settled exactly.
//
// The arithmetic is branch-free and mostly packed:
//   - u = h 2^-16, the 16-bit uniform, as (128 + h 2^-16) - 128, where the
//     float 128 + h 2^-16 is the bit pattern 0x4300 0000 | h (one byte
//     permute);
//   - RN(T) lands in the low bits of T + 1.5 * 2^23 (see sr_codes8 for the
//     sign);
//   - T - RN(T) is exact, and the largest of its eight magnitudes
//     certifies a group of eight at once.

__device__ __forceinline__ uint32_t prmt_bytes(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// min(a, b, c) with NaN propagated (a NaN position is never certified).
__device__ __forceinline__ float min3_nan(float a, float b, float c) {
  float r;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float min_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

constexpr uint32_t kSrMagic = 0x4B400000u;  // 1.5 * 2^23

// max(m, |a|, |b|) with NaN propagated.
__device__ __forceinline__ float max3_abs_nan(float m, float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
  return r;
}

// The stochastic codes of the eight elements x[0..7] (a multiple of eight
// apart from the tensor's start) from one Philox block r, by the certified
// rule above: element i draws the 16-bit half i & 1 (low first) of word
// i >> 1.  Returns the eight codes as nibbles, valid only when all eight are
// certified: that is when the returned largest distance |T - RN(T)| is
// below 1/2 - 2^-19 (NaN when an element is NaN); otherwise the caller
// settles all eight exactly.
//   RN(T) is formed as F1 = RN(T + 12582916) (1.5 * 2^23 + 4), and the code
// nibble as F1 - copysign(4, x): 1.5 * 2^23 + RN(T) for x >= 0, the same +8
// for x < 0, so the low nibble of its bits is the signed E2M1 code.  The
// nibbles are summed into the word by integer multiply-adds of the raw
// bits; the constant part of the bits (0x4B40 0000 at every nibble) is
// removed once.  A certified nibble is at most 15, so nothing carries.
__device__ __forceinline__ uint32_t sr_codes8(const float x[8], float inv, const Philox4& r,
                                              float& dmax) {
  const uint32_t words[4] = {r.x, r.y, r.z, r.w};
  uint32_t acc = 0u;
  float dm = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = 2 * k;
    const F2 ux{__uint_as_float(prmt_bytes(words[k], 0x43000000u, 0x7410u)),
                __uint_as_float(prmt_bytes(words[k], 0x43000000u, 0x7432u))};
    const F2 u = sub2(ux, F2{128.0f, 128.0f});                        // exact
    const F2 m{fabsf(__fmul_rn(x[i], inv)), fabsf(__fmul_rn(x[i + 1], inv))};
    const F2 p2 = fma2(m, F2{2.0f, 2.0f}, F2{0.5f, 0.5f});
    const F2 p1 = add2(m, F2{2.5f, 2.5f});
    const F2 ph = fma2(m, F2{0.5f, 0.5f}, F2{4.5f, 4.5f});
    const F2 sh{min_nan(min3_nan(p2.x, p1.x, ph.x), 7.5f), min_nan(min3_nan(p2.y, p1.y, ph.y), 7.5f)};
    const F2 T = sub2(sh, u);
    const F2 F1 = add2(T, F2{12582916.0f, 12582916.0f});
    const F2 d = sub2(T, sub2(F1, F2{12582916.0f, 12582916.0f}));
    dm = max3_abs_nan(dm, d.x, d.y);
    const F2 sg{__uint_as_float((__float_as_uint(x[i]) & 0x80000000u) | 0x40800000u),
                __uint_as_float((__float_as_uint(x[i + 1]) & 0x80000000u) | 0x40800000u)};
    const F2 F = sub2(F1, sg);
    acc += __float_as_uint(F.x) * (1u << (4 * i));
    acc += __float_as_uint(F.y) * (1u << (4 * i + 4));
  }
  dmax = dm;
  return acc - kSrMagic * 0x11111111u;
}

// Settling a bracket that straddles a rounding midpoint, without dividing.
// The two bracket codes are the neighbours lo < hi around the midpoint M of
// their values, and |x| / y lies within 2^-20 of M.  Then
// r = RN(M * y - |x|) is exact (M * y and |x| are multiples of a common
// quantum at most 2^7 apart), and q = RN(|x| / y) equals M exactly when |r|
// is at most y times half an ulp of M on the side of q (half an ulp below a
// power of two is half as large; at that bound the tie goes to M, whose
// significand is even).  So the code is the even one of lo and hi when
// q == M, lo when M * y > |x|, hi otherwise; no division, and exact.
__device__ __forceinline__ uint32_t settle_midpoint(float ax, float y, float M, uint32_t lo,
                                                    uint32_t hi) {
  const float r = __fmaf_rn(M, y, -ax);
  const uint32_t mb = __float_as_uint(M);
  const uint32_t half_bits = ((mb >> 23) - 24u) << 23;      // 2^(exponent(M) - 24)
  const bool pow2 = (mb & 0x7FFFFFu) == 0u;
  float half = __fmul_rn(y, __uint_as_float(half_bits));
  if (pow2 && r > 0.0f) half = __fmul_rn(half, 0.5f);
  if (fabsf(r) <= half) return (lo & 1u) ? hi : lo;
  return r > 0.0f ? lo : hi;
}

// e4m3 block scale code RN_e4m3(RN(bmax / den6)) through the certified
// bracket, settled exactly when the bracket straddles an e4m3 midpoint.
__device__ __forceinline__ uint32_t block_scale_code(float bmax, const ScaleDiv& sd) {
  const uint32_t lh = cvt_e4m3x2(__fmul_rn(bmax, sd.r_lo), __fmul_rn(bmax, sd.r_hi));
  uint32_t sb = lh & 0xFFu;
  if (sd.r_lo == 0.0f || sb != (lh >> 8)) {
    const uint32_t hb = lh >> 8;
    if (sd.r_lo != 0.0f && hb == sb + 1u && sd.den6 >= 0x1p-100f) {
      const float M = __fmul_rn(__fadd_rn(e4m3_value(sb), e4m3_value(hb)), 0.5f);
      sb = settle_midpoint(bmax, sd.den6, M, sb, hb);
    } else {
      sb = exact_e4m3_quotient(bmax, sd.den6);
    }
  }
  return sb;
}

// The multipliers of the E2M1 bracket for a decoded block scale eff:
// RN(RN(1/eff) * (1 -+ 2^-21)), both 0 when eff is 0 (the codes are then
// those of x * 0).  Certified only for eff in [2^-125, 2^125].
struct Bracket {
  float il, ih;
};

__device__ __forceinline__ Bracket make_bracket(float eff) {
  const float inv = __frcp_rn(eff);
  const bool zero = eff == 0.0f;
  return Bracket{zero ? 0.0f : __fmul_rn(inv, 0x1.fffffp-1f),    // 1 - 2^-21
                 zero ? 0.0f : __fmul_rn(inv, 0x1.000008p+0f)};  // 1 + 2^-21
}

__device__ __forceinline__ bool bracket_certified(float eff) {
  return eff == 0.0f || (eff >= 0x1p-125f && eff <= 0x1p125f);
}

// The E2M1 code of RN(x / eff) for eff in [2^-125, 2^125] when the bracket
// codes cl and ch of x differ.
__device__ __forceinline__ uint32_t settle_e2m1(float x, float eff, uint32_t cl, uint32_t ch) {
  const uint32_t ml = cl & 7u;
  if ((ch & 7u) == ml + 1u && (ch & 8u) == (cl & 8u) && eff >= 0x1p-100f) {
    const float M = __fmul_rn(__fadd_rn(e2m1_value(ml), e2m1_value(ml + 1u)), 0.5f);
    return (cl & 8u) | settle_midpoint(fabsf(x), eff, M, ml, ml + 1u);
  }
  return exact_e2m1_quotient(x, eff);
}

// max(0, |v[i]|) over a block (a NaN element is ignored, as by fmaxf), as a
// tree of three-input maxima.
__device__ __forceinline__ float absmax16(const float v[16]) {
  float a[5];
#pragma unroll
  for (int k = 0; k < 5; ++k) a[k] = max3_abs(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  return max3(max3(a[0], a[1], a[2]), max3(a[3], a[4], fabsf(v[15])), 0.0f);
}

// Quantize one block v[16] (residual already added) under tensor scale s_t.
// Writes the 8 packed bytes as two words, returns the e4m3 scale byte, and
// (kEF) leaves the dequantized values in q[16].
template <bool kSR, bool kEF>
__device__ __forceinline__ uint32_t quantize_block(const float v[16], float s_t, const ScaleDiv& sd,
                                                   uint64_t g0, uint32_t key0, uint32_t key1,
                                                   uint32_t step0, uint32_t step1, uint2& out,
                                                   float q[16]) {
  const float bmax = absmax16(v);
  const uint32_t sb = block_scale_code(bmax, sd);
  const float eff = __fmul_rn(e4m3_value(sb), s_t);
  uint32_t w0, w1;
  if (kSR) {
    // codes by sr_codes8, eight elements per Philox block at counter
    // (g0 >> 3) + k; the few uncertified elements (and every element when
    // eff is outside the certified range) take the exact division
    // afterwards, their random half drawn again
    const bool fast = eff >= 0x1p-125f && eff <= 0x1p125f;
    const float inv = fast ? rcp_rn(eff) : 0.0f;
    uint32_t pend = 0u;  // bit i: element i still to settle
    uint32_t ww[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint64_t oct = (g0 >> 3) + (uint64_t)k;
      const Philox4 r = philox4x32_10((uint32_t)oct, (uint32_t)(oct >> 32), step0, step1, key0,
                                      key1);
      float dmax;
      ww[k] = sr_codes8(v + 8 * k, inv, r, dmax);
      pend |= (fast && dmax < 0.5f - 0x1p-19f ? 0u : 0xFFu) << (8 * k);
    }
    w0 = ww[0];
    w1 = ww[1];
    while (pend != 0u) {
      const int i = __ffs(pend) - 1;
      pend &= pend - 1u;
      // element i by a tree of selects on its index bits
      const bool b0 = i & 1, b1 = i & 2, b2 = i & 4, b3 = i & 8;
      float e[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) e[t] = b0 ? v[2 * t + 1] : v[2 * t];
#pragma unroll
      for (int t = 0; t < 4; ++t) e[t] = b1 ? e[2 * t + 1] : e[2 * t];
#pragma unroll
      for (int t = 0; t < 2; ++t) e[t] = b2 ? e[2 * t + 1] : e[2 * t];
      const float xi = b3 ? e[1] : e[0];
      const uint64_t oct = (g0 >> 3) + (uint64_t)(i >> 3);
      const Philox4 r = philox4x32_10((uint32_t)oct, (uint32_t)(oct >> 32), step0, step1, key0,
                                      key1);
      const int j = (i >> 1) & 3;
      const uint32_t wj = j == 0 ? r.x : j == 1 ? r.y : j == 2 ? r.z : r.w;
      const uint32_t rwi = (i & 1) ? (wj & 0xFFFF0000u) : (wj << 16);
      const uint32_t code = exact_e2m1_sr_quotient(xi, eff, rwi);
      const int sh = 4 * (i & 7);
      if (i < 8)
        w0 = (w0 & ~(0xFu << sh)) | (code << sh);
      else
        w1 = (w1 & ~(0xFu << sh)) | (code << sh);
    }
  } else if (eff >= 0x1p-125f && eff <= 0x1p125f) {
    // RTN codes of RN(v / eff) through the certified bracket, 8 at a time
    const float inv = rcp_rn(eff);
    const float il = __fmul_rn(inv, 0x1.fffffp-1f);   // 1 - 2^-21
    const float ih = __fmul_rn(inv, 0x1.000008p+0f);  // 1 + 2^-21
    uint32_t lo[2], hi[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float* x = v + 8 * h;
      lo[h] = cvt_e2m1x8(__fmul_rn(x[0], il), __fmul_rn(x[1], il), __fmul_rn(x[2], il),
                         __fmul_rn(x[3], il), __fmul_rn(x[4], il), __fmul_rn(x[5], il),
                         __fmul_rn(x[6], il), __fmul_rn(x[7], il));
      hi[h] = cvt_e2m1x8(__fmul_rn(x[0], ih), __fmul_rn(x[1], ih), __fmul_rn(x[2], ih),
                         __fmul_rn(x[3], ih), __fmul_rn(x[4], ih), __fmul_rn(x[5], ih),
                         __fmul_rn(x[6], ih), __fmul_rn(x[7], ih));
    }
    w0 = lo[0];
    w1 = lo[1];
    // Elements whose two bracket codes differ (a few per thousand: quotients
    // on or next to an E2M1 rounding midpoint, many of them exact ties for
    // bf16 weights) are settled one at a time.
    uint32_t p0 = lo[0] ^ hi[0], p1 = lo[1] ^ hi[1];  // nibbles still to settle
    while ((p0 | p1) != 0u) {
      {
        const bool first = p0 != 0u;
        const uint32_t p = first ? p0 : p1;
        const int i = (__ffs(p) - 1) >> 2;
        const float* x = first ? v : v + 8;
        float xi = x[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) xi = (i == k) ? x[k] : xi;
        const uint32_t cl = ((first ? w0 : w1) >> (4 * i)) & 0xFu;
        const uint32_t ch = ((first ? hi[0] : hi[1]) >> (4 * i)) & 0xFu;
        const uint32_t code = settle_e2m1(xi, eff, cl, ch);
        const uint32_t c = code << (4 * i);
        const uint32_t m = 0xFu << (4 * i);
        if (first) {
          w0 = (w0 & ~m) | c;
          p0 &= ~m;
        } else {
          w1 = (w1 & ~m) | c;
          p1 &= ~m;
        }
      }
    }
  } else {
    // zero, tiny or huge decoded scale: exact division throughout
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = (eff == 0.0f) ? __fmul_rn(v[i], 0.0f) : __fdiv_rn(v[i], eff);
    w0 = cvt_e2m1x8(a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7]);
    w1 = cvt_e2m1x8(a[8], a[9], a[10], a[11], a[12], a[13], a[14], a[15]);
  }
  out = make_uint2(w0, w1);
  if (kEF) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(e2m1_value(w0 >> (4 * i)), eff);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[8 + i] = __fmul_rn(e2m1_value(w1 >> (4 * i)), eff);
  }
  return sb;
}

// Per-tensor constants of the E2M1 step for every e4m3 block-scale byte sb:
// the bracket multipliers of the decoded scale eff = RN(e4m3(sb) * s_t),
// eff itself, and flags: bit 0 the bracket is certified for eff, bit 1 eff
// is short (short_divisor).  One table of kEffEntries serves a warp for a
// whole tensor, so a block's E2M1 constants cost one shared-memory load
// instead of a decode, a multiply and a correctly rounded reciprocal.
struct alignas(16) EffEntry {
  float il, ih, eff;
  uint32_t flags;
};
constexpr int kEffEntries = 128;  // every byte with the sign bit clear

// The calling warp fills tab[0 .. kEffEntries) for tensor scale s_t.  The
// leading __syncwarp lets the table be refilled for another tensor after
// the warp's last reads of the old one.
__device__ __forceinline__ void build_eff_table(EffEntry* tab, float s_t) {
  const uint32_t lane = threadIdx.x & 31u;
  __syncwarp();
#pragma unroll
  for (int k = 0; k < kEffEntries / 32; ++k) {
    const uint32_t sb = lane + 32u * k;
    const float eff = __fmul_rn(e4m3_value(sb), s_t);
    const Bracket br = make_bracket(eff);
    EffEntry e;
    e.il = br.il;
    e.ih = br.ih;
    e.eff = eff;
    e.flags = (bracket_certified(eff) ? 1u : 0u) | (short_divisor(eff) ? 2u : 0u);
    tab[sb] = e;
  }
  __syncwarp();
}

// max(|a|, |b|) of each bf16 half; the sign bits of the result are junk.
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Round-to-nearest quantization of one block of 16 bf16 values (raw: the
// block's 8 words, element 2i in the low half of word i; no residual): the
// result of quantize_block<false, false>, faster.  The block maximum is
// taken on the bf16 pairs, the 32 bracket products are packed pairs, and
// the E2M1 constants come from the warp's table.  Bracket disagreements
// under a short divisor are exact ties and take the even code branch-free
// (short_divisor); the rest (near ties under a full-precision decoded scale,
// about one element in a thousand, or a scale outside the certified range)
// are settled one element at a time from the bracket codes already at hand.
__device__ __forceinline__ uint32_t quantize_block_bf16_rtn(const U32x8& raw, const ScaleDiv& sd,
                                                            const EffEntry* tab, uint2& out) {
  const uint32_t m = max_abs_bf16x2(
      max_abs_bf16x2(max_abs_bf16x2(raw.w[0], raw.w[1]), max_abs_bf16x2(raw.w[2], raw.w[3])),
      max_abs_bf16x2(max_abs_bf16x2(raw.w[4], raw.w[5]), max_abs_bf16x2(raw.w[6], raw.w[7])));
  const float bmax = fmaxf(bf16_lo(m & 0x7FFFu), bf16_hi(m & 0x7FFF0000u));
  uint32_t sb;
  if (sd.short6) {
    const uint32_t lh = cvt_e4m3x2(__fmul_rn(bmax, sd.r_lo), __fmul_rn(bmax, sd.r_hi));
    sb = lh & 0xFFu;
    sb += (sb ^ (lh >> 8)) & sb & 1u;  // a tie: the even code
  } else {
    sb = block_scale_code(bmax, sd);
  }
  const EffEntry e = tab[sb & (kEffEntries - 1)];
  const F2 kl{e.il, e.il}, kh{e.ih, e.ih};
  F2 pl[8], ph[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const F2 x{bf16_lo(raw.w[i]), bf16_hi(raw.w[i])};
    pl[i] = mul2(x, kl);
    ph[i] = mul2(x, kh);
  }
  uint32_t lo[2], hi[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const F2* a = pl + 4 * h;
    const F2* b = ph + 4 * h;
    lo[h] = cvt_e2m1x8(a[0].x, a[0].y, a[1].x, a[1].y, a[2].x, a[2].y, a[3].x, a[3].y);
    hi[h] = cvt_e2m1x8(b[0].x, b[0].y, b[1].x, b[1].y, b[2].x, b[2].y, b[3].x, b[3].y);
  }
  const bool cert = (e.flags & 1u) != 0u;
  uint32_t w[2], p[2];
  if (e.flags == 3u) {
    // ties: a differing nibble is lo's magnitude + 1, and the even code is
    // lo + 1 exactly when lo's magnitude is odd (it is at most 5)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      w[h] = lo[h] + ((lo[h] ^ hi[h]) & lo[h] & 0x11111111u);
      p[h] = 0u;
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      w[h] = lo[h];
      p[h] = cert ? lo[h] ^ hi[h] : 0xFFFFFFFFu;
    }
  }
  while ((p[0] | p[1]) != 0u) {
    const bool first = p[0] != 0u;
    const uint32_t pend = first ? p[0] : p[1];
    const int sh = (__ffs(pend) - 1) & ~3;  // the nibble of the element
    const int i = sh >> 2;                  // element i of the half
    // word (first ? 0 : 4) + i / 2 of the block, by a tree of selects
    const bool b0 = (i & 2) != 0, b1 = (i & 4) != 0;
    const uint32_t q0 = b0 ? raw.w[1] : raw.w[0], q1 = b0 ? raw.w[3] : raw.w[2];
    const uint32_t q2 = b0 ? raw.w[5] : raw.w[4], q3 = b0 ? raw.w[7] : raw.w[6];
    const uint32_t h0 = b1 ? q1 : q0, h1 = b1 ? q3 : q2;
    const uint32_t word = first ? h0 : h1;
    const float xi = (i & 1) ? bf16_hi(word) : bf16_lo(word);
    uint32_t code;
    if (cert)
      code = settle_e2m1(xi, e.eff, ((first ? lo[0] : lo[1]) >> sh) & 0xFu,
                         ((first ? hi[0] : hi[1]) >> sh) & 0xFu);
    else
      code = exact_e2m1_quotient(xi, e.eff);
    const uint32_t mk = 0xFu << sh;
    if (first) {
      w[0] = (w[0] & ~mk) | (code << sh);
      p[0] &= ~mk;
    } else {
      w[1] = (w[1] & ~mk) | (code << sh);
      p[1] &= ~mk;
    }
  }
  out = make_uint2(w[0], w[1]);
  return sb;
}

template <bool kBF16Out>
__device__ __forceinline__ void dequantize_store(uint32_t w0, uint32_t w1, float eff, void* y,
                                                 int64_t b) {
  float o[16];
  e2m1x8_to_f32(w0, o);
  e2m1x8_to_f32(w1, o + 8);
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = __fmul_rn(o[i], eff);
  if (kBF16Out) {
    U32x8 w;
#pragma unroll
    for (int i = 0; i < 8; ++i) w.w[i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
    st_v8(static_cast<uint16_t*>(y) + 16 * b, w);
  } else {
    store_f32x16(static_cast<float*>(y) + 16 * b, o);
  }
}


// Where the block scales of a [rows, 16 * cols] matrix go in the blocked
// layout (common.cuh).  A thread keeps its block's place as the byte offset
// of its row tile, the row inside the tile and the scale column, and steps
// it by the grid stride with adds and compares only: no division and no
// 64-bit multiply per block.  cols < 2^24 keeps every offset inside a row
// tile below 2^31.
struct BlockedMap {
  int64_t rows, cols, col_tiles;
};

struct BlockedCursor {
  int64_t base;  // (row / 128) * col_tiles * 512
  uint32_t rr;   // row % 128
  uint32_t c;    // scale column
};

struct BlockedStep {
  int64_t base;            // (stride rows / 128) * col_tiles * 512
  int64_t tile_row_bytes;  // col_tiles * 512
  uint32_t rr, c, cols;    // stride rows % 128, stride columns, cols
};

// a / d for a >= 0, d > 0; by 32-bit division when both fit (every weight
// matrix of the workloads), the 64-bit form costing several times more.
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int64_t d) {
  if (((a | d) >> 32) == 0) return (int64_t)((uint32_t)a / (uint32_t)d);
  return a / d;
}

__device__ __forceinline__ BlockedCursor blocked_cursor(int64_t b, const BlockedMap& bm) {
  const int64_t row = div_nonneg(b, bm.cols);
  return BlockedCursor{(row >> 7) * bm.col_tiles * 512, (uint32_t)(row & 127),
                       (uint32_t)(b - row * bm.cols)};
}

__device__ __forceinline__ BlockedStep blocked_step(int64_t stride, const BlockedMap& bm) {
  const int64_t rows = div_nonneg(stride, bm.cols);
  return BlockedStep{(rows >> 7) * bm.col_tiles * 512, bm.col_tiles * 512,
                     (uint32_t)(rows & 127), (uint32_t)(stride - rows * bm.cols),
                     (uint32_t)bm.cols};
}

// Byte offset of the cursor's scale: its row tile, then inside the tile the
// column tile, the row group (row / 32), the row within it and the column
// within the 4-byte word, which occupy disjoint bits.
__device__ __forceinline__ int64_t blocked_at(const BlockedCursor& q) {
  return q.base + (int64_t)(((q.c & ~3u) << 7) | ((q.rr & 31u) << 4) | ((q.rr >> 5) << 2) |
                            (q.c & 3u));
}

__device__ __forceinline__ void blocked_advance(BlockedCursor& q, const BlockedStep& st) {
  q.c += st.c;
  const bool wrap = q.c >= st.cols;
  q.c = wrap ? q.c - st.cols : q.c;
  q.rr += st.rr + (wrap ? 1u : 0u);
  const bool tile = q.rr >= 128u;
  q.rr = tile ? q.rr - 128u : q.rr;
  q.base += st.base + (tile ? st.tile_row_bytes : 0);
}

// Raw inputs of one block: x (one 256-bit word of bf16, two of fp32) and,
// with error feedback, the residual (two words).
template <bool kBF16, bool kRes>
struct BlockIn {
  U32x8 x[kBF16 ? 1 : 2];
  U32x8 r[kRes ? 2 : 1];
};

template <bool kBF16, bool kRes>
__device__ __forceinline__ void issue_block(const void* x, const float* residual, int64_t b,
                                            int64_t nblocks, BlockIn<kBF16, kRes>& in) {
  if (b < nblocks) {
    const uint8_t* xb = static_cast<const uint8_t*>(x) + b * (kBF16 ? 32 : 64);
    in.x[0] = ld_stream_v8(xb);
    if (!kBF16) in.x[kBF16 ? 0 : 1] = ld_stream_v8(xb + 32);
    if (kRes) {
      in.r[0] = ld_v8(residual + 16 * b);
      in.r[kRes ? 1 : 0] = ld_v8(residual + 16 * b + 8);
    }
  }
}

// The 16 values of a block (bf16 or fp32 x, plus the residual with error
// feedback, one fp32 addition each) from its raw words.
template <bool kBF16, bool kRes>
__device__ __forceinline__ void unpack_block(const BlockIn<kBF16, kRes>& in, float v[16],
                                             float r[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (kBF16) {
      v[2 * i] = bf16_lo(in.x[0].w[i]);
      v[2 * i + 1] = bf16_hi(in.x[0].w[i]);
    } else {
      v[i] = __uint_as_float(in.x[0].w[i]);
      v[8 + i] = __uint_as_float(in.x[kBF16 ? 0 : 1].w[i]);
    }
  }
  if (kRes) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r[i] = __uint_as_float(in.r[0].w[i]);
      r[8 + i] = __uint_as_float(in.r[kRes ? 1 : 0].w[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fadd_rn(v[i], r[i]);
  }
}

}  // namespace
}  // namespace fp4
