// scaled.cu -- E2M1 with one fp32 scale for a whole tensor.
//
// [WP2] "Block scaling" ("Why not one scale for the whole matrix?") and
// "Sixteen values aren't enough": the comparison points of block scaling.
// Codes are RN_e2m1(RN(x / s)) with one correctly rounded division per
// element; s = 1 rounds straight to FP4.  Dequantize: value(code) * s.
// The scale is a host value, or is read from the device: the one-scale-per-
// matrix choice s = RN(amax / 6) is formed from a tensor amax in device
// memory (the largest magnitude lands on 6, the largest E2M1 value).
//
// One thread per 16 elements: one 256-bit load of bf16 (two of fp32), an
// 8-byte store of codes; the inverse reads 8 bytes and writes 32 (bf16) or
// 64 (fp32).
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"

namespace fp4 {
namespace {

constexpr int kThreads = 256;

// s = RN(amax / 6), or 1 when that is not finite and > 0 (amax 0, say).
__device__ __forceinline__ float scale_from_amax(float amax) {
  const float s = __fdiv_rn(amax, 6.0f);
  return (s > 0.0f && s <= 3.40282347e38f) ? s : 1.0f;
}

// amax == NULL: the scale is s; otherwise s = scale_from_amax(*amax), which
// the first thread also writes to *scale_out.
template <bool kBF16>
__global__ void __launch_bounds__(kThreads)
    scaled_quantize_kernel(const void* __restrict__ x, int64_t nunits, float s,
                           const float* __restrict__ amax, float* __restrict__ scale_out,
                           uint8_t* __restrict__ packed) {
  if (amax) {
    s = scale_from_amax(*amax);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;
  }
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < nunits; u += stride) {
    float v[16];
    if (kBF16) {
      const U32x8 r = ld_stream_v8(static_cast<const uint16_t*>(x) + 16 * u);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(r.w[i]);
        v[2 * i + 1] = bf16_hi(r.w[i]);
      }
    } else {
      const float* p = static_cast<const float*>(x) + 16 * u;
      const U32x8 a = ld_stream_v8(p), b = ld_stream_v8(p + 8);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = __uint_as_float(a.w[i]);
        v[8 + i] = __uint_as_float(b.w[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fdiv_rn(v[i], s);
    const uint32_t w0 = cvt_e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
    const uint32_t w1 = cvt_e2m1x8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
    *reinterpret_cast<uint2*>(packed + 8 * u) = make_uint2(w0, w1);
  }
}

// s_dev != NULL: the scale is *s_dev instead of s.
template <bool kBF16Out>
__global__ void __launch_bounds__(kThreads)
    scaled_dequantize_kernel(const uint8_t* __restrict__ packed, int64_t nunits, float s,
                             const float* __restrict__ s_dev, void* __restrict__ y) {
  if (s_dev) s = *s_dev;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < nunits; u += stride) {
    const uint2 p = ld_stream_v2(packed + 8 * u);
    const uint32_t words[2] = {p.x, p.y};
    float o[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      e2m1x8_to_f32(words[h], o + 8 * h);
#pragma unroll
      for (int k = 0; k < 8; ++k) o[8 * h + k] = __fmul_rn(o[8 * h + k], s);
    }
    if (kBF16Out) {
      U32x8 w;
#pragma unroll
      for (int i = 0; i < 8; ++i) w.w[i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
      st_v8(static_cast<uint16_t*>(y) + 16 * u, w);
    } else {
      float* out = static_cast<float*>(y) + 16 * u;
      U32x8 a, b;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a.w[i] = __float_as_uint(o[i]);
        b.w[i] = __float_as_uint(o[8 + i]);
      }
      st_v8(out, a);
      st_v8(out + 8, b);
    }
  }
}

bool scale_ok(float s) { return s > 0.0f && s <= 3.40282347e38f; }

fp4_status launch_scaled_quantize(const void* x, int dtype, int64_t n, float scale,
                                  const float* amax, float* scale_out, uint8_t* packed,
                                  cudaStream_t s) {
  const int64_t nu = n / 16;
  if (dtype == FP4_BF16)
    return launch<scaled_quantize_kernel<true>>(nu, kThreads, 0, s, x, nu, scale, amax,
                                                scale_out, packed);
  return launch<scaled_quantize_kernel<false>>(nu, kThreads, 0, s, x, nu, scale, amax, scale_out,
                                               packed);
}

fp4_status launch_scaled_dequantize(const uint8_t* packed, int64_t n, float scale,
                                    const float* s_dev, void* y, int out_dtype, cudaStream_t s) {
  const int64_t nu = n / 16;
  if (out_dtype == FP4_BF16)
    return launch<scaled_dequantize_kernel<true>>(nu, kThreads, 0, s, packed, nu, scale, s_dev, y);
  return launch<scaled_dequantize_kernel<false>>(nu, kThreads, 0, s, packed, nu, scale, s_dev, y);
}

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

fp4_status fp4_scaled_quantize(const void* x, int dtype, int64_t n, float scale, uint8_t* packed,
                               void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!scale_ok(scale)) return FP4_ERR_ARG;
  if (n > 0 && (!x || !packed)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(packed, 8)) return FP4_ERR_ALIGN;
  if (n == 0) return FP4_OK;
  return launch_scaled_quantize(x, dtype, n, scale, nullptr, nullptr, packed, as_stream(stream));
}

fp4_status fp4_scaled_quantize_amax(const void* x, int dtype, int64_t n, const float* amax,
                                    float* scale_out, uint8_t* packed, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!amax || !scale_out || (n > 0 && (!x || !packed))) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(packed, 8) || !aligned(amax, 4) || !aligned(scale_out, 4))
    return FP4_ERR_ALIGN;
  // an empty tensor still publishes its scale: one CTA, no units
  return launch_scaled_quantize(x, dtype, n, 1.0f, amax, scale_out, packed, as_stream(stream));
}

fp4_status fp4_scaled_dequantize(const uint8_t* packed, int64_t n, float scale, void* y,
                                 int out_dtype, void* stream) {
  if (!dtype_ok(out_dtype)) return FP4_ERR_DTYPE;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!scale_ok(scale)) return FP4_ERR_ARG;
  if (n > 0 && (!packed || !y)) return FP4_ERR_NULL;
  if (!aligned(packed, 8) || !aligned(y, 32)) return FP4_ERR_ALIGN;
  if (n == 0) return FP4_OK;
  return launch_scaled_dequantize(packed, n, scale, nullptr, y, out_dtype, as_stream(stream));
}

fp4_status fp4_scaled_dequantize_dev(const uint8_t* packed, int64_t n, const float* scale,
                                     void* y, int out_dtype, void* stream) {
  if (!dtype_ok(out_dtype)) return FP4_ERR_DTYPE;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!scale || (n > 0 && (!packed || !y))) return FP4_ERR_NULL;
  if (!aligned(packed, 8) || !aligned(y, 32) || !aligned(scale, 4)) return FP4_ERR_ALIGN;
  if (n == 0) return FP4_OK;
  return launch_scaled_dequantize(packed, n, 1.0f, scale, y, out_dtype, as_stream(stream));
}

}  // extern "C"
