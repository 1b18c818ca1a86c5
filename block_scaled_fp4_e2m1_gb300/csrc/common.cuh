// common.cuh -- device helpers shared by the codec kernels (sm_103a).
//
// All arithmetic that decides a code is written with explicit round-to-
// nearest intrinsics (__fmul_rn, __fadd_rn, __fdiv_rn, __frcp_rn, __fsqrt_rn)
// and the library is built with -fmad=false, so no multiply-add is ever
// contracted: each operation is one correctly rounded fp32 operation.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp4codec.h"

namespace fp4 {

// ------------------------------------------------------------ memory access

struct U32x8 {
  uint32_t w[8];
};

// 256-bit read-only load that does not allocate in L1 (streamed input).
__device__ __forceinline__ U32x8 ld_stream_v8(const void* p) {
  U32x8 r;
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                 "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(p));
  return r;
}

// 256-bit load of data this kernel may also write (no .nc).
__device__ __forceinline__ U32x8 ld_v8(const void* p) {
  U32x8 r;
  asm volatile("ld.global.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                 "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v8(void* p, const U32x8& v) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// ---------------------------------------------------- asynchronous staging
//
// Group bookkeeping of cp.async copies into shared memory (the copies
// themselves are issued where they are used).

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// max(|a|, |b|, |c|) and max(a, b, c) in one three-input max (exact; the
// order of a max does not matter; a NaN operand is ignored).
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The 8 codes of w (code i in bits 4i+3..4i) as exact floats, through the
// hardware e2m1x2 -> f16x2 conversion of each byte of w.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float o[8]) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(o[2 * k]), "=f"(o[2 * k + 1])
        : "r"(h[k]));
  }
}

// ------------------------------------------------------ packed fp32 pairs
//
// Two fp32 values in one 64-bit register pair, operated on by the packed
// add / sub / mul / fma.rn.f32x2 instructions: each lane is one correctly
// rounded fp32 operation, identical to the scalar .rn form, at one issue
// slot for both.  Unlike the scalar .rn forms, a packed multiply whose
// result feeds a packed addition can be fused into one fma by the compiler
// (measured on sm_103a), so callers form such products with scalar
// multiplies.

struct F2 {
  float x, y;
};

__device__ __forceinline__ F2 add2(F2 a, F2 b) {
  F2 r;
  asm("{.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ F2 sub2(F2 a, F2 b) {
  F2 r;
  asm("{.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
  F2 r;
  asm("{.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
  F2 r;
  asm("{.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// ------------------------------------------------------------ bf16 <-> f32

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats to a bf16 pair, round to nearest-even; lo in bits 15:0.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// --------------------------------------------------------------------- E2M1

// Round-to-nearest-even, saturating E2M1 encode of two floats; lo -> bits 3:0.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Eight floats to eight E2M1 codes (round-to-nearest-even, saturating) in one
// 32-bit word, a[i] in bits 4i+3..4i.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float a0, float a1, float a2, float a3, float a4,
                                               float a5, float a6, float a7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
  return r;
}

// Two floats to two E4M3 bytes (round-to-nearest-even, saturating): lo in
// bits 7:0, hi in bits 15:8.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Exact value of the E2M1 code in bits 3:0 of c: sign to bit 31, the three
// magnitude bits to bits 24:22 of a binary32 pattern, which reads as
// value * 2^-126 (a subnormal for 0.5); one exact multiply by 2^126 restores
// the value.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  uint32_t bits = ((c & 8u) << 28) | ((c & 7u) << 22);
  return __fmul_rn(__uint_as_float(bits), 0x1p126f);
}

// --------------------------------------------------------------------- E4M3

// Round-to-nearest-even, saturating E4M3 (OCP E4M3FN) encode of one float.
__device__ __forceinline__ uint32_t cvt_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return (uint32_t)(r & 0xFFu);
}

// Exact value of an E4M3FN byte (through f16, which holds every E4M3 value).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  uint32_t h2;
  uint16_t in = (uint16_t)(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  uint16_t h = (uint16_t)(h2 & 0xFFFFu);
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}

// --------------------------------------------------------------- Philox4x32

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11): per round
// the products of counter words 0 and 2 with the two multipliers are split
// into high and low halves; the high halves are XORed with counter words 1
// and 3 and the key; the key advances by the two Weyl increments.
struct Philox4 {
  uint32_t x, y, z, w;
};

// The 64-bit product of two 32-bit words as one wide multiply.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
  asm("{\n\t.reg .b64 p;\n\tmul.wide.u32 p, %2, %3;\n\tmov.b64 {%1, %0}, p;\n\t}"
      : "=r"(hi), "=r"(lo)
      : "r"(a), "r"(b));
}

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                  uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi1, lo1;
    mul_wide(0xD2511F53u, c0, hi0, lo0);
    mul_wide(0xCD9E8D57u, c2, hi1, lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return Philox4{c0, c1, c2, c3};
}

// Stochastic E2M1 encode of a with the random word rw (a 16-bit uniform h
// as h << 16): between grid neighbours lo <= |a| < hi the upper one is taken
// iff (rw >> 8) * 2^-24 = h * 2^-16 < (|a| - lo) / (hi - lo); |a| >= 6
// gives 6.
__device__ __forceinline__ uint32_t e2m1_sr(float a, uint32_t rw) {
  uint32_t sign = (__float_as_uint(a) >> 28) & 8u;
  float m = fabsf(a);
  if (!(m < 6.0f)) return (m >= 6.0f) ? (sign | 7u) : 0u;  // NaN -> 0
  uint32_t c = (uint32_t)(m >= 0.5f) + (uint32_t)(m >= 1.0f) + (uint32_t)(m >= 1.5f) +
               (uint32_t)(m >= 2.0f) + (uint32_t)(m >= 3.0f) + (uint32_t)(m >= 4.0f);
  float lo = e2m1_value(c);
  // 1 / (hi - lo): 2 below 2, 1 in [2, 4), 0.5 in [4, 6)
  float k = __uint_as_float((128u - (uint32_t)(c >= 4u) - (uint32_t)(c >= 6u)) << 23);
  float frac = __fmul_rn(__fsub_rn(m, lo), k);
  float u = __fmul_rn((float)(rw >> 8), 0x1p-24f);
  return sign | (c + (uint32_t)(u < frac));
}

// ---------------------------------------------------- blocked scale layout
// The layout of block scales that Blackwell block-scaled tensor-core matmuls
// read: a [rows, cols] matrix of one-byte scales, zero-padded to whole tiles
// of 128 rows x 4 columns, tiles stored in row-major order, 512 bytes each;
// scale (r, c) of a tile at byte 16 (r mod 32) + 4 floor(r / 32) + c.

// Byte offset of scale (r, c) of the padded matrix; col_tiles = ceil(cols/4).
__device__ __forceinline__ int64_t blocked_offset(int64_t r, int64_t c, int64_t col_tiles) {
  return ((((r >> 7) * col_tiles) + (c >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) +
         (c & 3);
}

// Zero the padding bytes of a blocked buffer: columns cols .. 4 col_tiles - 1
// of every row, then every column of rows rows .. 128 ceil(rows/128) - 1.
// Threads t = 0, stride, 2 stride, ... share the work.
__device__ __forceinline__ void blocked_zero_padding(uint8_t* out, int64_t rows, int64_t cols,
                                                     int64_t col_tiles, int64_t t,
                                                     int64_t stride) {
  const int64_t pc = 4 * col_tiles - cols;               // padded columns, 0..3
  const int64_t pw = 4 * col_tiles;                      // padded row width
  const int64_t n1 = rows * pc;
  const int64_t n2 = (((rows + 127) >> 7) * 128 - rows) * pw;
  for (int64_t i = t; i < n1 + n2; i += stride) {
    int64_t r, c;
    if (i < n1) {
      r = i / pc;
      c = cols + (i - r * pc);
    } else {
      const int64_t j = i - n1, q = j / pw;
      r = rows + q;
      c = j - q * pw;
    }
    out[blocked_offset(r, c, col_tiles)] = 0;
  }
}

// ------------------------------------------------------------- reductions

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  return __reduce_max_sync(0xFFFFFFFFu, v);
}

}  // namespace fp4
