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
// Layout: a thread owns 16 consecutive elements of a group (one 256-bit
// load of bf16), so a group of G spans G/16 consecutive lanes (4, 8 or 16)
// and never leaves its warp: no shared memory and no CTA barrier.
//   - sum of squares: a balanced pairwise tree over adjacent elements, first
//     inside the thread (16 -> 1), then across lanes by xor-shuffle 1, 2, ...;
//   - transform: butterfly stages h = 1, 2, 4, 8 inside the thread, stages
//     h = 16, 32, ... across lanes (lane xor h/16), in the natural
//     (Sylvester) order; the lower partner keeps a + b, the upper a - b,
//     computed as one correctly rounded fma(+-1, own, partner);
//   - each thread packs its 16 codes into 8 bytes and stores them directly.
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

// Normalized Walsh-Hadamard transform of the group whose elements
// 16*(lane % (G/16)) .. +15 this thread holds in y[].
template <int G>
__device__ __forceinline__ void wht_group(float y[16], int lane) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const float a = y[i], b = y[i + h];
      y[i] = __fadd_rn(a, b);
      y[i + h] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int m = 1; m < G / 16; m <<= 1) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;  // upper partner: partner - own
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float p = __shfl_xor_sync(0xFFFFFFFFu, y[i], m);
      y[i] = __fmaf_rn(sgn, y[i], p);
    }
  }
  const float c = wht_norm<G>();
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(y[i], c);
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int m = 1; m < G / 16; m <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int m = 1; m < G / 16; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

template <bool kBF16>
__device__ __forceinline__ void load16(const void* x, int64_t u, float v[16]) {
  if (kBF16) {
    U32x8 r = ld_stream_v8(static_cast<const uint16_t*>(x) + 16 * u);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(r.w[i]);
      v[2 * i + 1] = bf16_hi(r.w[i]);
    }
  } else {
    const float* p = static_cast<const float*>(x) + 16 * u;
    U32x8 a = ld_stream_v8(p), b = ld_stream_v8(p + 8);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = __uint_as_float(a.w[i]);
      v[8 + i] = __uint_as_float(b.w[i]);
    }
  }
}

// Units are 16-element chunks; the loop is warp-uniform so that every lane
// takes part in the shuffles, and lanes past the end compute on zeros
// without storing (the chunk count is a multiple of G/16, so a group is
// either entirely inside or entirely past the end).
template <int G, bool kBF16>
__global__ void __launch_bounds__(kThreads)
    encode_kernel(const void* __restrict__ x, int64_t nchunks, uint8_t* __restrict__ packed,
                  float* __restrict__ s1_out, float* __restrict__ s2_out) {
  constexpr int LPG = G / 16;
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t u0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31); u0 < nchunks; u0 += stride) {
    const int64_t u = u0 + lane;
    const bool valid = u < nchunks;
    float y[16];
    if (valid) {
      load16<kBF16>(x, u, y);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = 0.0f;
    }
    // RMS scale
    float sq[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) sq[i] = __fmul_rn(y[i], y[i]);
#pragma unroll
    for (int w = 16; w > 1; w >>= 1) {
#pragma unroll
      for (int i = 0; i < w / 2; ++i) sq[i] = __fadd_rn(sq[2 * i], sq[2 * i + 1]);
    }
    const float ss = group_sum<G>(sq[0]);
    const float rms = __fsqrt_rn(__fmul_rn(ss, 1.0f / (float)G));
    const float inv1 = rms == 0.0f ? 0.0f : __frcp_rn(rms);
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(y[i], inv1);
    // transform
    wht_group<G>(y, lane);
    // absmax scale into [-6, 6]
    float zmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) zmax = fmaxf(zmax, fabsf(y[i]));
    zmax = group_max<G>(zmax);
    const float sc2 = __fdiv_rn(zmax, 6.0f);
    const float inv2 = sc2 == 0.0f ? 0.0f : __frcp_rn(sc2);
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w0 |= cvt_e2m1x2(__fmul_rn(y[2 * i], inv2), __fmul_rn(y[2 * i + 1], inv2)) << (8 * i);
      w1 |= cvt_e2m1x2(__fmul_rn(y[8 + 2 * i], inv2), __fmul_rn(y[8 + 2 * i + 1], inv2)) << (8 * i);
    }
    if (valid) {
      *reinterpret_cast<uint2*>(packed + 8 * u) = make_uint2(w0, w1);
      if ((lane & (LPG - 1)) == 0) {
        s1_out[u / LPG] = rms;
        s2_out[u / LPG] = sc2;
      }
    }
  }
}

template <int G, bool kBF16Out>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const uint8_t* __restrict__ packed, const float* __restrict__ s1_in,
                  const float* __restrict__ s2_in, int64_t nchunks, void* __restrict__ out) {
  constexpr int LPG = G / 16;
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t u0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31); u0 < nchunks; u0 += stride) {
    const int64_t u = u0 + lane;
    const bool valid = u < nchunks;
    uint2 p = make_uint2(0u, 0u);
    float sc1 = 0.0f, sc2 = 0.0f;
    if (valid) {
      p = ld_stream_v2(packed + 8 * u);
      sc1 = s1_in[u / LPG];
      sc2 = s2_in[u / LPG];
    }
    float z[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      z[i] = __fmul_rn(e2m1_value(p.x >> (4 * i)), sc2);
      z[8 + i] = __fmul_rn(e2m1_value(p.y >> (4 * i)), sc2);
    }
    wht_group<G>(z, lane);
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = __fmul_rn(z[i], sc1);
    if (valid) {
      if (kBF16Out) {
        U32x8 w;
#pragma unroll
        for (int i = 0; i < 8; ++i) w.w[i] = pack_bf16x2(z[2 * i], z[2 * i + 1]);
        st_v8(static_cast<uint16_t*>(out) + 16 * u, w);
      } else {
        float* o = static_cast<float*>(out) + 16 * u;
        U32x8 a, b;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          a.w[i] = __float_as_uint(z[i]);
          b.w[i] = __float_as_uint(z[8 + i]);
        }
        st_v8(o, a);
        st_v8(o + 8, b);
      }
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
  const int64_t nchunks = rows * cols / 16;
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
  const int64_t nchunks = rows * cols / 16;
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
