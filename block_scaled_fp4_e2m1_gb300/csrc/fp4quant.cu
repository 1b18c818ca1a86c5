// fp4quant.cu -- FP4Quant group encode / decode.
//
// [FP4Quant] "Why four bits need more than rounding": each contiguous group
// gets an RMS scale, then a normalized Walsh-Hadamard transform made of
// additions and subtractions, then an absmax scale into the E2M1 range; both
// scales travel with the codes.  "Making compression cheap enough to help":
// the transform exchanges values between the threads of a warp by register
// shuffles, codes are paired and packed two per byte in registers, and the
// receiver unpacks, dequantizes and runs the inverse transform.
//
// Layout: a thread owns 32 consecutive elements of a group (two 256-bit
// loads of bf16), so a group of G spans G/32 consecutive lanes (2, 4 or 8)
// and never leaves its warp: no shared memory and no CTA barrier.
//   - sum of squares: a balanced pairwise tree over adjacent elements, first
//     inside the thread (32 -> 1), then across lanes by xor-shuffle 1, 2, ...;
//   - transform: butterfly stages h = 1 .. 16 inside the thread, stages
//     h = 32, 64, ... across lanes (lane xor h/32), in the natural
//     (Sylvester) order; the lower partner keeps a + b, the upper a - b,
//     computed as one correctly rounded fma(+-1, own, partner).  Holding 32
//     elements keeps one more stage inside the thread than 16 would: the
//     shuffles, which bound these kernels, drop by a quarter to a half;
//   - each thread packs its 32 codes into 16 bytes and stores them directly.
// The arithmetic order (reciprocal scales, the tree, the stage order) is the
// one the CPU oracle follows, so codes and scales are bit-exact.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"

namespace fp4 {
namespace {

constexpr int kThreads = 256;

template <int G>
__device__ __forceinline__ float wht_norm() {
  // RN(1/sqrt(G)): 1/8, RN(sqrt(2)/16) = 0x3DB504F3, 1/16
  return G == 64 ? 0.125f : (G == 256 ? 0.0625f : __uint_as_float(0x3DB504F3u));
}

// A thread's 32 elements as 16 packed pairs P[i] = (y[i], y[i + 16]), so
// that the butterfly stages h = 1 .. 8, the cross-lane stages and the final
// scalings run two elements per instruction; stage h = 16 pairs the two
// halves of each P[i].  A product that feeds an addition is always formed
// by a scalar multiply: the compiler may fuse a packed multiply into the
// packed addition that consumes it (one rounding instead of two), which
// would break the exact operation order.
constexpr int kE = 32;  // elements per thread

struct Row32 {
  F2 p[16];
  __device__ __forceinline__ float& at(int i) { return i < 16 ? p[i].x : p[i - 16].y; }
};

__device__ __forceinline__ F2 splat(float v) { return F2{v, v}; }

// Normalized Walsh-Hadamard transform of the group whose elements
// 32*(lane % (G/32)) .. +31 this thread holds.
template <int G>
__device__ __forceinline__ void wht_group(Row32& y, int lane) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const F2 a = y.p[i], b = y.p[i + h];
      y.p[i] = add2(a, b);
      y.p[i + h] = sub2(a, b);
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // h = 16
    const float a = y.p[i].x, b = y.p[i].y;
    y.p[i] = F2{__fadd_rn(a, b), __fsub_rn(a, b)};
  }
#pragma unroll
  for (int m = 1; m < G / kE; m <<= 1) {
    const F2 sgn = splat((lane & m) ? -1.0f : 1.0f);  // upper partner: partner - own
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const F2 q{__shfl_xor_sync(0xFFFFFFFFu, y.p[i].x, m),
                 __shfl_xor_sync(0xFFFFFFFFu, y.p[i].y, m)};
      y.p[i] = fma2(sgn, y.p[i], q);
    }
  }
  const F2 c = splat(wht_norm<G>());
#pragma unroll
  for (int i = 0; i < 16; ++i) y.p[i] = mul2(y.p[i], c);
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int m = 1; m < G / kE; m <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int m = 1; m < G / kE; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

template <bool kBF16>
__device__ __forceinline__ void load32(const void* x, int64_t u, Row32& y) {
  if (kBF16) {
    const uint16_t* p = static_cast<const uint16_t*>(x) + kE * u;
    const U32x8 a = ld_stream_v8(p), b = ld_stream_v8(p + 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y.p[2 * i].x = bf16_lo(a.w[i]);
      y.p[2 * i + 1].x = bf16_hi(a.w[i]);
      y.p[2 * i].y = bf16_lo(b.w[i]);
      y.p[2 * i + 1].y = bf16_hi(b.w[i]);
    }
  } else {
    const float* p = static_cast<const float*>(x) + kE * u;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const U32x8 a = ld_stream_v8(p + 8 * k), b = ld_stream_v8(p + 16 + 8 * k);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        y.p[8 * k + i].x = __uint_as_float(a.w[i]);
        y.p[8 * k + i].y = __uint_as_float(b.w[i]);
      }
    }
  }
}

// The raw words of a chunk, fetched one grid-stride step ahead of their use
// so that a thread's next loads are in flight while it transforms the
// current chunk (bf16 input: two 256-bit words; fp32 input is loaded when
// used, four words would cost too many registers).
struct RawBF16 {
  U32x8 a, b;
};

__device__ __forceinline__ void fetch_bf16(const void* x, int64_t u, bool ok, RawBF16& r) {
  if (ok) {
    const uint16_t* p = static_cast<const uint16_t*>(x) + kE * u;
    r.a = ld_stream_v8(p);
    r.b = ld_stream_v8(p + 16);
  }
}

__device__ __forceinline__ void unpack_bf16(const RawBF16& r, bool ok, Row32& y) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    y.p[2 * i].x = ok ? bf16_lo(r.a.w[i]) : 0.0f;
    y.p[2 * i + 1].x = ok ? bf16_hi(r.a.w[i]) : 0.0f;
    y.p[2 * i].y = ok ? bf16_lo(r.b.w[i]) : 0.0f;
    y.p[2 * i + 1].y = ok ? bf16_hi(r.b.w[i]) : 0.0f;
  }
}

// Units are 32-element chunks; the loop is warp-uniform so that every lane
// takes part in the shuffles, and lanes past the end compute on zeros
// without storing (the chunk count is a multiple of G/32, so a group is
// either entirely inside or entirely past the end).
// Encodes the chunk u (32 elements in y) and stores its codes and, from the
// group's first lane, its two scales.
template <int G>
__device__ __forceinline__ void encode_chunk(Row32& y, int64_t u, bool valid, int lane,
                                             uint8_t* __restrict__ packed,
                                             float* __restrict__ s1_out,
                                             float* __restrict__ s2_out) {
  constexpr int LPG = G / kE;
  // RMS scale: the pairwise tree over adjacent squares, levels 1-4 two
  // sums per instruction ((0..15 | 16..31) halves side by side)
  F2 sq[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    sq[i] = F2{__fmul_rn(y.p[i].x, y.p[i].x), __fmul_rn(y.p[i].y, y.p[i].y)};
#pragma unroll
  for (int w = 16; w > 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w / 2; ++i) sq[i] = add2(sq[2 * i], sq[2 * i + 1]);
  }
  const float ss = group_sum<G>(__fadd_rn(sq[0].x, sq[0].y));
  const float rms = __fsqrt_rn(__fmul_rn(ss, 1.0f / (float)G));
  const float inv1 = rms == 0.0f ? 0.0f : __frcp_rn(rms);
#pragma unroll
  for (int i = 0; i < 16; ++i) y.p[i] = F2{__fmul_rn(y.p[i].x, inv1), __fmul_rn(y.p[i].y, inv1)};
  // transform
  wht_group<G>(y, lane);
  // absmax scale into [-6, 6]
  float zmax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) zmax = fmaxf(zmax, fmaxf(fabsf(y.p[i].x), fabsf(y.p[i].y)));
  zmax = group_max<G>(zmax);
  const float sc2 = __fdiv_rn(zmax, 6.0f);
  const F2 inv2 = splat(sc2 == 0.0f ? 0.0f : __frcp_rn(sc2));
#pragma unroll
  for (int i = 0; i < 16; ++i) y.p[i] = mul2(y.p[i], inv2);
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] = cvt_e2m1x8(y.at(8 * k), y.at(8 * k + 1), y.at(8 * k + 2), y.at(8 * k + 3),
                      y.at(8 * k + 4), y.at(8 * k + 5), y.at(8 * k + 6), y.at(8 * k + 7));
  if (valid) {
    *reinterpret_cast<uint4*>(packed + 16 * u) = make_uint4(w[0], w[1], w[2], w[3]);
    if ((lane & (LPG - 1)) == 0) {
      s1_out[u / LPG] = rms;
      s2_out[u / LPG] = sc2;
    }
  }
}

// bf16 input keeps the next chunk's loads in flight (a two-buffer ring
// walked by an unrolled loop, so no registers are copied); fp32 input loads
// each chunk when it is used.
template <int G, bool kBF16>
__global__ void __launch_bounds__(kThreads, kBF16 ? 2 : 3)
    encode_kernel(const void* __restrict__ x, int64_t nchunks, uint8_t* __restrict__ packed,
                  float* __restrict__ s1_out, float* __restrict__ s2_out) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t u0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31);
  if (kBF16) {
    RawBF16 ring[2];
    fetch_bf16(x, u0 + lane, u0 + lane < nchunks, ring[0]);
    for (;;) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (u0 >= nchunks) return;
        const int64_t u = u0 + lane;
        fetch_bf16(x, u + stride, u + stride < nchunks, ring[s ^ 1]);
        Row32 y;
        unpack_bf16(ring[s], u < nchunks, y);
        encode_chunk<G>(y, u, u < nchunks, lane, packed, s1_out, s2_out);
        u0 += stride;
      }
    }
  } else {
    for (; u0 < nchunks; u0 += stride) {
      const int64_t u = u0 + lane;
      const bool valid = u < nchunks;
      Row32 y;
      if (valid) {
        load32<false>(x, u, y);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) y.p[i] = splat(0.0f);
      }
      encode_chunk<G>(y, u, valid, lane, packed, s1_out, s2_out);
    }
  }
}

// The 8 codes of w (code i in bits 4i+3..4i) as exact floats, through the
// hardware e2m1x2 -> f16x2 conversion.
__device__ __forceinline__ void e2m1x8_values(uint32_t w, float o[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t h2;
    const uint16_t byte = (uint16_t)((w >> (8 * k)) & 0xFFu);
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u16 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
        : "=r"(h2)
        : "h"(byte));
    const uint16_t lo = (uint16_t)(h2 & 0xFFFFu), hi = (uint16_t)(h2 >> 16);
    asm("cvt.f32.f16 %0, %1;" : "=f"(o[2 * k]) : "h"(lo));
    asm("cvt.f32.f16 %0, %1;" : "=f"(o[2 * k + 1]) : "h"(hi));
  }
}

// A chunk's codes and its group's two scales.
struct DecIn {
  uint4 p;
  float sc1, sc2;
};

template <int G>
__device__ __forceinline__ void fetch_dec(const uint8_t* __restrict__ packed,
                                          const float* __restrict__ s1_in,
                                          const float* __restrict__ s2_in, int64_t u, bool ok,
                                          DecIn& d) {
  constexpr int LPG = G / kE;
  if (ok) {
    d.p = ld_stream_v4(packed + 16 * u);
    d.sc1 = s1_in[u / LPG];
    d.sc2 = s2_in[u / LPG];
  } else {
    d.p = make_uint4(0u, 0u, 0u, 0u);
    d.sc1 = d.sc2 = 0.0f;
  }
}

// The next chunk's codes and scales are in flight while the current one is
// decoded (a two-buffer ring walked by an unrolled loop).
template <int G, bool kBF16Out>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const uint8_t* __restrict__ packed, const float* __restrict__ s1_in,
                  const float* __restrict__ s2_in, int64_t nchunks, void* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t u0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31);
  DecIn ring[2];
  fetch_dec<G>(packed, s1_in, s2_in, u0 + lane, u0 + lane < nchunks, ring[0]);
  for (;;) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (u0 >= nchunks) return;
      const int64_t u = u0 + lane;
      const bool valid = u < nchunks;
      fetch_dec<G>(packed, s1_in, s2_in, u + stride, u + stride < nchunks, ring[s ^ 1]);
      const DecIn& d = ring[s];
      float v[32];
      e2m1x8_values(d.p.x, v);
      e2m1x8_values(d.p.y, v + 8);
      e2m1x8_values(d.p.z, v + 16);
      e2m1x8_values(d.p.w, v + 24);
      Row32 z;
#pragma unroll
      for (int i = 0; i < 16; ++i) z.p[i] = F2{__fmul_rn(v[i], d.sc2), __fmul_rn(v[i + 16], d.sc2)};
      wht_group<G>(z, lane);
      const F2 m1 = splat(d.sc1);
#pragma unroll
      for (int i = 0; i < 16; ++i) z.p[i] = mul2(z.p[i], m1);
      if (valid) {
        if (kBF16Out) {
          uint16_t* o = static_cast<uint16_t*>(out) + kE * u;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            U32x8 w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w.w[i] = pack_bf16x2(z.at(16 * k + 2 * i), z.at(16 * k + 2 * i + 1));
            st_v8(o + 16 * k, w);
          }
        } else {
          float* o = static_cast<float*>(out) + kE * u;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            U32x8 w;
#pragma unroll
            for (int i = 0; i < 8; ++i) w.w[i] = __float_as_uint(z.at(8 * k + i));
            st_v8(o + 8 * k, w);
          }
        }
      }
      u0 += stride;
    }
  }
}

template <int G>
fp4_status launch_encode(const void* x, int dtype, int64_t nchunks, uint8_t* packed, float* s1,
                         float* s2, cudaStream_t s) {
  if (dtype == FP4_BF16)
    return launch<encode_kernel<G, true>>(nchunks, kThreads, 0, s, x, nchunks, packed, s1, s2);
  return launch<encode_kernel<G, false>>(nchunks, kThreads, 0, s, x, nchunks, packed, s1, s2);
}

template <int G>
fp4_status launch_decode(const uint8_t* packed, const float* s1, const float* s2, int64_t nchunks,
                         void* y, int dtype, cudaStream_t s) {
  if (dtype == FP4_BF16)
    return launch<decode_kernel<G, true>>(nchunks, kThreads, 0, s, packed, s1, s2, nchunks, y);
  return launch<decode_kernel<G, false>>(nchunks, kThreads, 0, s, packed, s1, s2, nchunks, y);
}

bool group_ok(int g) { return g == 64 || g == 128 || g == 256; }

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

fp4_status fp4quant_encode(const void* x, int dtype, int64_t rows, int64_t cols, int group,
                           uint8_t* packed, float* s1, float* s2, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (!group_ok(group)) return FP4_ERR_ARG;
  if (rows < 0 || cols < 0 || cols % group != 0) return FP4_ERR_SHAPE;
  const int64_t nchunks = rows * cols / kE;
  if (nchunks > 0 && (!x || !packed || !s1 || !s2)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(packed, 16) || !aligned(s1, 4) || !aligned(s2, 4))
    return FP4_ERR_ALIGN;
  if (nchunks == 0) return FP4_OK;
  cudaStream_t s = as_stream(stream);
  if (group == 64) return launch_encode<64>(x, dtype, nchunks, packed, s1, s2, s);
  if (group == 128) return launch_encode<128>(x, dtype, nchunks, packed, s1, s2, s);
  return launch_encode<256>(x, dtype, nchunks, packed, s1, s2, s);
}

fp4_status fp4quant_decode(const uint8_t* packed, const float* s1, const float* s2, int64_t rows,
                           int64_t cols, int group, void* y, int out_dtype, void* stream) {
  if (!dtype_ok(out_dtype)) return FP4_ERR_DTYPE;
  if (!group_ok(group)) return FP4_ERR_ARG;
  if (rows < 0 || cols < 0 || cols % group != 0) return FP4_ERR_SHAPE;
  const int64_t nchunks = rows * cols / kE;
  if (nchunks > 0 && (!y || !packed || !s1 || !s2)) return FP4_ERR_NULL;
  if (!aligned(y, 32) || !aligned(packed, 16) || !aligned(s1, 4) || !aligned(s2, 4))
    return FP4_ERR_ALIGN;
  if (nchunks == 0) return FP4_OK;
  cudaStream_t s = as_stream(stream);
  if (group == 64) return launch_decode<64>(packed, s1, s2, nchunks, y, out_dtype, s);
  if (group == 128) return launch_decode<128>(packed, s1, s2, nchunks, y, out_dtype, s);
  return launch_decode<256>(packed, s1, s2, nchunks, y, out_dtype, s);
}

}  // extern "C"
