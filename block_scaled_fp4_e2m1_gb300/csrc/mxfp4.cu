// mxfp4.cu -- MXFP4 quantize (BF16ToFP4Row).
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
    float bmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
    // floor(log2 bmax) = biased exponent - 127 (subnormal and zero clamp below)
    int e = (int)((__float_as_uint(bmax) >> 23) & 0xFFu) - 129;
    e = e < -127 ? -127 : e;
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-E, a normal float
    uint32_t w[4];
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
    *reinterpret_cast<uint4*>(packed + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
    scales[b] = (uint8_t)(e + 127);
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
