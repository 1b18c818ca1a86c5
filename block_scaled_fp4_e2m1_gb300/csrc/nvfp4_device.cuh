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

#include "common.cuh"

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

template <bool kBF16>
__device__ __forceinline__ void load_block(const void* x, int64_t b, float v[16]) {
  if (kBF16) {
    U32x8 r = ld_stream_v8(static_cast<const uint16_t*>(x) + 16 * b);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(r.w[i]);
      v[2 * i + 1] = bf16_hi(r.w[i]);
    }
  } else {
    const float* p = static_cast<const float*>(x) + 16 * b;
    U32x8 a = ld_stream_v8(p), c = ld_stream_v8(p + 8);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = __uint_as_float(a.w[i]);
      v[8 + i] = __uint_as_float(c.w[i]);
    }
  }
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

// Per-kernel constants of the block-scale division u = bmax / den6.
struct ScaleDiv {
  float den6;    // 6 * s_t
  float r_lo;    // RN(RN(1/den6) * (1 - 2^-21)), 0 when den6 is outside [2^-125, 2^125]
  float r_hi;    // RN(RN(1/den6) * (1 + 2^-21))
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

// Quantize one block v[16] (residual already added) under tensor scale s_t.
// Writes the 8 packed bytes as two words, returns the e4m3 scale byte, and
// (kEF) leaves the dequantized values in q[16].
template <bool kSR, bool kEF>
__device__ __forceinline__ uint32_t quantize_block(const float v[16], float s_t, const ScaleDiv& sd,
                                                   uint64_t g0, uint32_t key0, uint32_t key1,
                                                   uint32_t step0, uint32_t step1, uint2& out,
                                                   float q[16]) {
  float bmax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
  // e4m3 block scale RN_e4m3(RN(bmax / den6)), through the certified bracket
  uint32_t sb;
  {
    const uint32_t lh = cvt_e4m3x2(__fmul_rn(bmax, sd.r_lo), __fmul_rn(bmax, sd.r_hi));
    sb = lh & 0xFFu;
    if (sd.r_lo == 0.0f || sb != (lh >> 8)) {
      // the bracket straddles the e4m3 midpoint between codes sb and sb + 1
      const uint32_t hb = lh >> 8;
      if (sd.r_lo != 0.0f && hb == sb + 1u && sd.den6 >= 0x1p-100f) {
        const float M = __fmul_rn(__fadd_rn(e4m3_value(sb), e4m3_value(hb)), 0.5f);
        sb = settle_midpoint(bmax, sd.den6, M, sb, hb);
      } else {
        sb = exact_e4m3_quotient(bmax, sd.den6);
      }
    }
  }
  const float eff = __fmul_rn(e4m3_value(sb), s_t);
  uint32_t w0, w1;
  if (kSR) {
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = (eff == 0.0f) ? __fmul_rn(v[i], 0.0f) : __fdiv_rn(v[i], eff);
    uint32_t codes[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint64_t quad = (g0 >> 2) + (uint64_t)k;
      Philox4 r = philox4x32_10((uint32_t)quad, (uint32_t)(quad >> 32), step0, step1, key0, key1);
      codes[4 * k + 0] = e2m1_sr(a[4 * k + 0], r.x);
      codes[4 * k + 1] = e2m1_sr(a[4 * k + 1], r.y);
      codes[4 * k + 2] = e2m1_sr(a[4 * k + 2], r.z);
      codes[4 * k + 3] = e2m1_sr(a[4 * k + 3], r.w);
    }
    w0 = w1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w0 |= codes[i] << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) w1 |= codes[8 + i] << (4 * i);
  } else if (eff >= 0x1p-125f && eff <= 0x1p125f) {
    // RTN codes of RN(v / eff) through the certified bracket, 8 at a time
    const float inv = __frcp_rn(eff);
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
    // Only the elements whose two bracket codes differ (a few per thousand,
    // quotients on or next to an E2M1 rounding midpoint) are divided; each
    // position is its own guarded call so a warp pays only for the positions
    // some lane needs.
    uint32_t p0 = lo[0] ^ hi[0], p1 = lo[1] ^ hi[1];  // nibbles still to settle
    // Elements whose two bracket codes differ (a few per thousand: quotients
    // on or next to an E2M1 rounding midpoint, many of them exact ties for
    // bf16 weights) are settled one at a time.
    while ((p0 | p1) != 0u) {
      {
        const bool first = p0 != 0u;
        const uint32_t p = first ? p0 : p1;
        const int i = (__ffs(p) - 1) >> 2;
        const float* x = first ? v : v + 8;
        float xi = x[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) xi = (i == k) ? x[k] : xi;
        // the element's lo/hi codes straddle the E2M1 midpoint between
        // magnitudes ml and ml + 1
        const uint32_t cl = ((first ? w0 : w1) >> (4 * i)) & 0xFu;
        const uint32_t ch = ((first ? hi[0] : hi[1]) >> (4 * i)) & 0xFu;
        const uint32_t ml = cl & 7u;
        uint32_t code;
        if ((ch & 7u) == ml + 1u && (ch & 8u) == (cl & 8u) && eff >= 0x1p-100f) {
          const float M = __fmul_rn(__fadd_rn(e2m1_value(ml), e2m1_value(ml + 1u)), 0.5f);
          code = (cl & 8u) | settle_midpoint(fabsf(xi), eff, M, ml, ml + 1u);
        } else {
          code = exact_e2m1_quotient(xi, eff);
        }
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

// Decode the 8 codes of w (code i in bits 4i+3..4i) to exact floats via the
// hardware e2m1x2 -> f16x2 conversion.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float o[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t h2;
    const uint16_t byte = (uint16_t)((w >> (8 * k)) & 0xFFu);
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u16 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
        : "=r"(h2)
        : "h"(byte));
    uint16_t lo = (uint16_t)(h2 & 0xFFFFu), hi = (uint16_t)(h2 >> 16);
    asm("cvt.f32.f16 %0, %1;" : "=f"(o[2 * k]) : "h"(lo));
    asm("cvt.f32.f16 %0, %1;" : "=f"(o[2 * k + 1]) : "h"(hi));
  }
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

}  // namespace
}  // namespace fp4
