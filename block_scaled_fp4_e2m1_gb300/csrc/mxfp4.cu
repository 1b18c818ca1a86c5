// mxfp4.cu -- MXFP4 quantize (BF16ToFP4Row), and the backward-path pair:
// FP8 (E4M3, one fp32 scale per 128) -> MXFP4, and MXFP4 dequantize.
//
// [MoE-FP4] "方法概述" and "核心技术贡献" 2: activations become MXFP4 row by
// row, E2M1 elements with one UE8M0 scale per 32 elements ([WP2] "Block
// scaling": the scale is a power of two).  The exponent follows the OCP
// microscaling rule: E = floor(log2(block amax)) - 2, read from the exponent
// field of the block amax (no math library), clamped to [-127, 127]; codes
// are RN_e2m1(x * 2^-E), exact scaling, [6, 8) saturating to 6.
//
// Layout: rows are contiguous and cols % 32 == 0, so the 32-blocks of the
// whole tensor are contiguous in flat order and block b owns input elements
// 32b..32b+31, packed bytes 16b..16b+15 and scale byte b.  One thread owns
// one block per grid-stride step: two 256-bit loads of bf16 (four of fp32),
// one 128-bit store of codes, one scale byte.  HBM-bound.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"

namespace fp4 {
namespace {

constexpr int kThreads = 256;

// The MXFP4 block of 32 values: UE8M0 byte and 16 packed code bytes.
__device__ __forceinline__ uint32_t mxfp4_block(const float v[32], uint32_t w[4]) {
  float bmax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
  // floor(log2 bmax) = biased exponent - 127 (subnormal and zero clamp below)
  int e = (int)((__float_as_uint(bmax) >> 23) & 0xFFu) - 129;
  e = e < -127 ? -127 : e;
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-E, a normal float
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t acc = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 8 * k + 2 * i;
      acc |= cvt_e2m1x2(__fmul_rn(v[j], inv), __fmul_rn(v[j + 1], inv)) << (8 * i);
    }
    w[k] = acc;
  }
  return (uint32_t)(e + 127);
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads)
    mxfp4_quantize_kernel(const void* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ packed,
                          uint8_t* __restrict__ scales) {
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += stride) {
    float v[32];
    if (kBF16) {
      const uint16_t* p = static_cast<const uint16_t*>(x) + 32 * b;
      U32x8 r0 = ld_stream_v8(p), r1 = ld_stream_v8(p + 16);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(r0.w[i]);
        v[2 * i + 1] = bf16_hi(r0.w[i]);
        v[16 + 2 * i] = bf16_lo(r1.w[i]);
        v[16 + 2 * i + 1] = bf16_hi(r1.w[i]);
      }
    } else {
      const float* p = static_cast<const float*>(x) + 32 * b;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        U32x8 r = ld_stream_v8(p + 8 * k);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[8 * k + i] = __uint_as_float(r.w[i]);
      }
    }
    uint32_t w[4];
    const uint32_t sb = mxfp4_block(v, w);
    *reinterpret_cast<uint4*>(packed + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
    scales[b] = (uint8_t)sb;
  }
}

// Backward-path FP4 ([MoE-FP4] "局限与未来方向": the backward pass in FP4
// is future work; "方法概述": gradients travel in FP8).  One thread per
// 32-block: one 256-bit load of 32 E4M3 bytes, the block's fp32 scale (one
// per 128, shared by 4 threads), each value RN(e4m3 * scale) in fp32, then
// the MXFP4 block rule above.
__global__ void __launch_bounds__(kThreads)
    fp8_to_fp4_row_kernel(const uint8_t* __restrict__ fp8, const float* __restrict__ fp8_scales,
                          int64_t nblocks, uint8_t* __restrict__ packed,
                          uint8_t* __restrict__ scales) {
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += stride) {
    const U32x8 r = ld_stream_v8(fp8 + 32 * b);
    const float s = __ldg(fp8_scales + b / 4);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t h2;
        const uint16_t pair = (uint16_t)(r.w[i] >> (16 * h));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        float lo, hi;
        asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"((uint16_t)(h2 & 0xFFFFu)));
        asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"((uint16_t)(h2 >> 16)));
        v[4 * i + 2 * h] = __fmul_rn(lo, s);
        v[4 * i + 2 * h + 1] = __fmul_rn(hi, s);
      }
    }
    uint32_t w[4];
    const uint32_t sb = mxfp4_block(v, w);
    *reinterpret_cast<uint4*>(packed + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
    scales[b] = (uint8_t)sb;
  }
}

// MXFP4 dequantize: one thread per 32-block, 16 code bytes (128-bit load)
// and one scale byte in, 32 values out (256-bit stores).  value(code) is
// exact in f16 and fp32, and the scale 2^(S-127) is applied as one exact
// multiply.  S = 255 is the format's NaN: every value of the block is the
// quiet NaN 0x7FC00000 (bf16 0x7FC0).
template <bool kBF16Out>
__global__ void __launch_bounds__(kThreads)
    mxfp4_dequantize_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                            int64_t nblocks, void* __restrict__ y) {
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += stride) {
    const uint4 p = ld_stream_v4(packed + 16 * b);
    const uint32_t S = ld_stream_u8(scales + b);
    const float f = __uint_as_float(S == 0u ? 0x00400000u : (S << 23));  // 2^(S - 127)
    const uint32_t words[4] = {p.x, p.y, p.z, p.w};
    float o[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      e2m1x8_to_f32(words[k], o + 8 * k);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[8 * k + j] = __fmul_rn(o[8 * k + j], f);
    }
    const bool nan = S == 255u;
    if (kBF16Out) {
      uint16_t* out = static_cast<uint16_t*>(y) + 32 * b;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        U32x8 w;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w.w[i] = nan ? 0x7FC07FC0u : pack_bf16x2(o[16 * h + 2 * i], o[16 * h + 2 * i + 1]);
        st_v8(out + 16 * h, w);
      }
    } else {
      float* out = static_cast<float*>(y) + 32 * b;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        U32x8 w;
#pragma unroll
        for (int i = 0; i < 8; ++i) w.w[i] = nan ? 0x7FC00000u : __float_as_uint(o[8 * h + i]);
        st_v8(out + 8 * h, w);
      }
    }
  }
}

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" fp4_status mxfp4_quantize(const void* x, int dtype, int64_t rows, int64_t cols,
                                     uint8_t* packed, uint8_t* scales, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (rows < 0 || cols < 0 || cols % 32 != 0) return FP4_ERR_SHAPE;
  const int64_t nb = rows * (cols / 32);
  if (nb > 0 && (!x || !packed || !scales)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(packed, 16)) return FP4_ERR_ALIGN;
  if (nb == 0) return FP4_OK;
  cudaStream_t s = as_stream(stream);
  if (dtype == FP4_BF16)
    return launch<mxfp4_quantize_kernel<true>>(nb, kThreads, 0, s, x, nb, packed, scales);
  return launch<mxfp4_quantize_kernel<false>>(nb, kThreads, 0, s, x, nb, packed, scales);
}

extern "C" fp4_status fp8_to_fp4_row(const uint8_t* fp8, const float* fp8_scales, int64_t rows,
                                     int64_t cols, uint8_t* packed, uint8_t* scales,
                                     void* stream) {
  if (rows < 0 || cols < 0 || cols % 128 != 0) return FP4_ERR_SHAPE;
  const int64_t nb = rows * (cols / 32);
  if (nb > 0 && (!fp8 || !fp8_scales || !packed || !scales)) return FP4_ERR_NULL;
  if (!aligned(fp8, 32) || !aligned(fp8_scales, 4) || !aligned(packed, 16)) return FP4_ERR_ALIGN;
  if (nb == 0) return FP4_OK;
  return launch<fp8_to_fp4_row_kernel>(nb, kThreads, 0, as_stream(stream), fp8, fp8_scales, nb,
                                       packed, scales);
}

extern "C" fp4_status mxfp4_dequantize(const uint8_t* packed, const uint8_t* scales, int64_t rows,
                                       int64_t cols, void* y, int out_dtype, void* stream) {
  if (!dtype_ok(out_dtype)) return FP4_ERR_DTYPE;
  if (rows < 0 || cols < 0 || cols % 32 != 0) return FP4_ERR_SHAPE;
  const int64_t nb = rows * (cols / 32);
  if (nb > 0 && (!packed || !scales || !y)) return FP4_ERR_NULL;
  if (!aligned(packed, 16) || !aligned(y, 32)) return FP4_ERR_ALIGN;
  if (nb == 0) return FP4_OK;
  cudaStream_t s = as_stream(stream);
  if (out_dtype == FP4_BF16)
    return launch<mxfp4_dequantize_kernel<true>>(nb, kThreads, 0, s, packed, scales, nb, y);
  return launch<mxfp4_dequantize_kernel<false>>(nb, kThreads, 0, s, packed, scales, nb, y);
}
