// nvfp4.cu -- NVFP4 tensor amax, quantize (RTN / stochastic, optional error
// feedback), dequantize, and the fused training-step qdq.
//
// [fp4-train] "How it works": 16-element blocks, scale block_absmax / 6
// encoded to e4m3, every element divided by the decoded scale and encoded to
// E2M1 by round-to-nearest or by stochastic rounding from a counter-based
// (seed, step, global index) RNG, optional per-element error-feedback
// residual.  [WP2] "Block scaling": one fp32 scale per tensor besides the
// block scales (chosen as amax / (6 * 448)).
//
// Layout: one thread owns one 16-element block per grid-stride step: 32 B
// of bf16 (one 256-bit load) or 64 B of fp32 (two), 8 B of packed codes and
// 1 B of scale.  A warp's loads cover 1 or 2 KB of contiguous input, every
// 256-bit load one full 32-byte sector.  HBM-bound; no shared memory.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "host_common.h"
#include "nvfp4_device.cuh"

namespace fp4 {
namespace {

// Blocks handled by one thread per pass of the amax loop: their loads are
// all issued before any is used, which keeps 4 x 32 (bf16) or 4 x 64 (fp32)
// bytes per thread in flight.
constexpr int kAmaxUnroll = 4;

template <bool kBF16, bool kRes>
__global__ void __launch_bounds__(kThreads)
    amax_kernel(const void* __restrict__ x, const float* __restrict__ residual, int64_t nblocks,
                float* __restrict__ amax_ws) {
  constexpr int kWords = kBF16 ? 1 : 2;  // 256-bit loads per block of x
  float m = 0.0f;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t b0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; b0 < nblocks;
       b0 += kAmaxUnroll * stride) {
    U32x8 raw[kAmaxUnroll][kWords];
    U32x8 res[kRes ? kAmaxUnroll : 1][2];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      const int64_t b = b0 + u * stride;
#pragma unroll
      for (int k = 0; k < kWords; ++k) {
        if (b < nblocks) {
          raw[u][k] = ld_stream_v8(static_cast<const uint8_t*>(x) + (kBF16 ? 32 : 64) * b + 32 * k);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) raw[u][k].w[i] = 0u;
        }
      }
      if (kRes) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (b < nblocks) {
            res[u][k] = ld_stream_v8(residual + 16 * b + 8 * k);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) res[u][k].w[i] = 0u;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (kBF16) {
          v[2 * i] = bf16_lo(raw[u][0].w[i]);
          v[2 * i + 1] = bf16_hi(raw[u][0].w[i]);
        } else {
          v[i] = __uint_as_float(raw[u][0].w[i]);
          v[8 + i] = __uint_as_float(raw[u][kWords - 1].w[i]);
        }
      }
      if (kRes) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[i] = __fadd_rn(v[i], __uint_as_float(res[u][0].w[i]));
          v[8 + i] = __fadd_rn(v[8 + i], __uint_as_float(res[u][1].w[i]));
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    }
  }
  block_max_to(m, amax_ws);
}

// Blocks a thread keeps in flight ahead of the one it computes: the loads of
// the next kDepth blocks of its grid-stride sequence are issued before the
// current block is quantized, so HBM latency hides behind the arithmetic.
template <bool kBF16, bool kRes>
struct QuantPipe {
  static constexpr int kDepth = (kBF16 && !kRes) ? 2 : 1;
};

// CTAs of kThreads per SM that the register allocation must allow: 4 is 64
// registers a thread, 3 is 80, 2 is 128.  The blocked-scale cursor needs a
// few more registers than 64.
template <bool kBF16, bool kSR, bool kRes, bool kBlk>
constexpr int quantize_min_ctas() {
  return (kRes || kSR) ? 2 : ((!kBF16 || kBlk) ? 3 : 4);
}

// A thread quantizes one block per grid-stride step; the loads of the next
// kD blocks are in flight meanwhile.  The ring of kD + 1 buffers is walked
// by a fully unrolled inner loop, so every buffer index is a constant and no
// registers are copied.  bf16 round-to-nearest without error feedback takes
// quantize_block_bf16_rtn with its warp's table of E2M1 constants,
// everything else quantize_block.
//
// kBlk writes block b's scale at its place in the blocked layout instead of
// at byte b (a BlockedCursor per thread); the padding bytes are zeroed
// first.
template <bool kBF16, bool kSR, bool kRes, bool kBlk>
__global__ void __launch_bounds__(kThreads, quantize_min_ctas<kBF16, kSR, kRes, kBlk>())
    quantize_kernel(const void* __restrict__ x, float* __restrict__ residual, int64_t nblocks,
                    uint64_t seed, uint64_t step, int tscale_mode, float* __restrict__ tensor_scale,
                    const float* __restrict__ amax_ws, uint8_t* __restrict__ packed,
                    uint8_t* __restrict__ scales, BlockedMap bm) {
  constexpr int kD = QuantPipe<kBF16, kRes>::kDepth;
  constexpr bool kFast = kBF16 && !kSR && !kRes;
  __shared__ EffEntry eff_tabs[kFast ? (kThreads / 32) * kEffEntries : 1];
  float s_t;
  if (tscale_mode == FP4_TSCALE_GIVEN) {
    s_t = sanitize_scale(*tensor_scale);
  } else {
    s_t = tensor_scale_from_amax(*amax_ws);
    if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = s_t;
  }
  const ScaleDiv sd = make_scale_div(s_t);
  EffEntry* const tab = eff_tabs + (kFast ? (threadIdx.x >> 5) * kEffEntries : 0);
  if (kFast) build_eff_table(tab, s_t);
  const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
  const uint32_t st0 = (uint32_t)step, st1 = (uint32_t)(step >> 32);
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  BlockedCursor cur{0, 0u, 0u};
  BlockedStep cstep{0, 0, 0u, 0u, 1u};
  if (kBlk) {
    blocked_zero_padding(scales, bm.rows, bm.cols, bm.col_tiles, b, stride);
    if (bm.cols > 0) {
      cur = blocked_cursor(b, bm);
      cstep = blocked_step(stride, bm);
    }
  }

  BlockIn<kBF16, kRes> buf[kD + 1];
#pragma unroll
  for (int d = 0; d < kD; ++d) issue_block<kBF16, kRes>(x, residual, b + d * stride, nblocks, buf[d]);
  for (;;) {
#pragma unroll
    for (int s = 0; s <= kD; ++s) {
      if (b >= nblocks) return;
      issue_block<kBF16, kRes>(x, residual, b + kD * stride, nblocks, buf[(s + kD) % (kD + 1)]);
      uint2 out;
      uint32_t sb;
      float r[16], q[16];
      if (kFast) {
        sb = quantize_block_bf16_rtn(buf[s].x[0], sd, tab, out);
      } else {
        float v[16];
        unpack_block<kBF16, kRes>(buf[s], v, r);
        sb = quantize_block<kSR, kRes>(v, s_t, sd, (uint64_t)(16 * b), key0, key1, st0, st1, out,
                                       q);
        if (kRes) {
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __fsub_rn(v[i], q[i]);
        }
      }
      *reinterpret_cast<uint2*>(packed + 8 * b) = out;
      if (kBlk) {
        scales[blocked_at(cur)] = (uint8_t)sb;
        blocked_advance(cur, cstep);
      } else {
        scales[b] = (uint8_t)sb;
      }
      if (kRes) store_f32x16(residual + 16 * b, r);
      b += stride;
    }
  }
}

// A thread decodes units of two blocks (16 B of codes, 2 scale bytes, one
// 128-bit and one 16-bit load), two units per pass with all loads first.
// An odd last block is decoded alone.
template <bool kBF16Out>
__global__ void __launch_bounds__(kThreads)
    dequantize_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                      const float* __restrict__ tensor_scale, int64_t nblocks, void* __restrict__ y) {
  const float s_t = tensor_scale ? sanitize_scale(*tensor_scale) : 1.0f;
  const int64_t npairs = nblocks >> 1;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  for (int64_t p0 = tid; p0 < npairs; p0 += 2 * stride) {
    uint4 pk[2];
    uint32_t sc[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t p = p0 + u * stride;
      if (p < npairs) {
        pk[u] = ld_stream_v4(packed + 16 * p);
        uint16_t s2;
        asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(s2) : "l"(scales + 2 * p));
        sc[u] = s2;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t p = p0 + u * stride;
      if (p < npairs) {
        dequantize_store<kBF16Out>(pk[u].x, pk[u].y, __fmul_rn(e4m3_value(sc[u] & 0xFFu), s_t),
                                   y, 2 * p);
        dequantize_store<kBF16Out>(pk[u].z, pk[u].w, __fmul_rn(e4m3_value(sc[u] >> 8), s_t), y,
                                   2 * p + 1);
      }
    }
  }
  if ((nblocks & 1) && tid == 0) {
    const int64_t b = nblocks - 1;
    const uint2 q = ld_stream_v2(packed + 8 * b);
    dequantize_store<kBF16Out>(q.x, q.y, __fmul_rn(e4m3_value(ld_stream_u8(scales + b)), s_t), y, b);
  }
}

// v = ((W - lr*G) + r), each step one fp32 operation.
template <bool kG, bool kRes>
__device__ __forceinline__ void qdq_update(const uint16_t* w, const float* g, float lr,
                                           const float* residual, int64_t b, float v[16],
                                           float r[16], bool stream_res) {
  U32x8 wr = ld_v8(w + 16 * b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(wr.w[i]);
    v[2 * i + 1] = bf16_hi(wr.w[i]);
  }
  if (kG) {
    float gg[16];
    load_f32x16_stream(g + 16 * b, gg);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fsub_rn(v[i], __fmul_rn(lr, gg[i]));
  }
  if (kRes) {
    if (stream_res)
      load_f32x16_stream(residual + 16 * b, r);
    else
      load_f32x16(residual + 16 * b, r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fadd_rn(v[i], r[i]);
  }
}

template <bool kG, bool kRes>
__global__ void __launch_bounds__(kThreads)
    qdq_amax_kernel(const uint16_t* __restrict__ w, const float* __restrict__ g, float lr,
                    const float* __restrict__ residual, int64_t nblocks, float* __restrict__ amax_ws) {
  float m = 0.0f;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += stride) {
    float v[16], r[16];
    qdq_update<kG, kRes>(w, g, lr, residual, b, v, r, true);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  }
  block_max_to(m, amax_ws);
}

template <bool kG, bool kRes, bool kSR, bool kPacked>
__global__ void __launch_bounds__(kThreads)
    qdq_kernel(uint16_t* __restrict__ w, const float* __restrict__ g, float lr,
               float* __restrict__ residual, int64_t nblocks, uint64_t seed, uint64_t step,
               int tscale_mode, float* __restrict__ tensor_scale, const float* __restrict__ amax_ws,
               uint8_t* __restrict__ packed, uint8_t* __restrict__ scales) {
  float s_t;
  if (tscale_mode == FP4_TSCALE_GIVEN) {
    s_t = sanitize_scale(*tensor_scale);
  } else {
    s_t = tensor_scale_from_amax(*amax_ws);
    if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = s_t;
  }
  const ScaleDiv sd = make_scale_div(s_t);
  const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
  const uint32_t st0 = (uint32_t)step, st1 = (uint32_t)(step >> 32);
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const int lane = threadIdx.x & 31;
  // warp-uniform trip count (lanes past the end compute on zeros and store
  // nothing): measured faster than a per-thread bound for this kernel
  for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b - lane < nblocks; b += stride) {
    const bool valid = b < nblocks;
    float v[16], r[16], q[16];
    if (valid) {
      qdq_update<kG, kRes>(w, g, lr, residual, b, v, r, false);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = r[i] = 0.0f;
    }
    uint2 out;
    uint32_t sb = quantize_block<kSR, true>(v, s_t, sd, (uint64_t)(16 * b), key0, key1, st0, st1,
                                            out, q);
    if (!valid) continue;
    if (kPacked) {
      *reinterpret_cast<uint2*>(packed + 8 * b) = out;
      scales[b] = (uint8_t)sb;
    }
    U32x8 wo;
#pragma unroll
    for (int i = 0; i < 8; ++i) wo.w[i] = pack_bf16x2(q[2 * i], q[2 * i + 1]);
    st_v8(w + 16 * b, wo);
    if (kRes) {
#pragma unroll
      for (int i = 0; i < 16; ++i) r[i] = __fsub_rn(v[i], q[i]);
      store_f32x16(residual + 16 * b, r);
    }
  }
}

fp4_status launch_amax(const void* x, int dtype, int64_t n, const float* residual, float* amax_ws,
                       cudaStream_t s) {
  if (cudaMemsetAsync(amax_ws, 0, sizeof(float), s) != cudaSuccess) return FP4_ERR_CUDA;
  const int64_t nb = n / 16;
  if (nb == 0) return FP4_OK;
  const int64_t units = (nb + kAmaxUnroll - 1) / kAmaxUnroll;
  if (dtype == FP4_BF16) {
    if (residual) return launch<amax_kernel<true, true>>(units, kThreads, 0, s, x, residual, nb, amax_ws);
    return launch<amax_kernel<true, false>>(units, kThreads, 0, s, x, residual, nb, amax_ws);
  }
  if (residual) return launch<amax_kernel<false, true>>(units, kThreads, 0, s, x, residual, nb, amax_ws);
  return launch<amax_kernel<false, false>>(units, kThreads, 0, s, x, residual, nb, amax_ws);
}

template <bool kBF16, bool kSR, bool kRes, bool kBlk>
fp4_status launch_quantize_k(const void* x, int64_t nb, float* residual, uint64_t seed, uint64_t step,
                             int mode, float* ts, const float* amax, uint8_t* packed, uint8_t* scales,
                             const BlockedMap& bm, cudaStream_t s) {
  return launch<quantize_kernel<kBF16, kSR, kRes, kBlk>>(nb, kThreads, 0, s, x, residual, nb, seed,
                                                         step, mode, ts, amax, packed, scales, bm);
}

template <bool kBF16, bool kBlk>
fp4_status launch_quantize_t(const void* x, int64_t nb, float* residual, int rounding, uint64_t seed,
                             uint64_t step, int mode, float* ts, const float* amax, uint8_t* packed,
                             uint8_t* scales, const BlockedMap& bm, cudaStream_t s) {
  if (rounding == FP4_SR) {
    if (residual)
      return launch_quantize_k<kBF16, true, true, kBlk>(x, nb, residual, seed, step, mode, ts, amax,
                                                        packed, scales, bm, s);
    return launch_quantize_k<kBF16, true, false, kBlk>(x, nb, residual, seed, step, mode, ts, amax,
                                                       packed, scales, bm, s);
  }
  if (residual)
    return launch_quantize_k<kBF16, false, true, kBlk>(x, nb, residual, seed, step, mode, ts, amax,
                                                       packed, scales, bm, s);
  return launch_quantize_k<kBF16, false, false, kBlk>(x, nb, residual, seed, step, mode, ts, amax,
                                                      packed, scales, bm, s);
}

// The shared part of nvfp4_quantize and nvfp4_quantize_blocked after the
// argument checks: the amax pass in COMPUTE mode, then the quantize launch.
template <bool kBlk>
fp4_status quantize_common(const void* x, int dtype, int64_t n, float* residual, int rounding,
                           uint64_t seed, uint64_t step, int tscale_mode, float* tensor_scale,
                           float* amax_ws, uint8_t* packed, uint8_t* scales, const BlockedMap& bm,
                           cudaStream_t s) {
  if (tscale_mode == FP4_TSCALE_COMPUTE) {
    fp4_status st = launch_amax(x, dtype, n, residual, amax_ws, s);
    if (st != FP4_OK) return st;
  }
  const int64_t nb = n / 16;
  // An empty tensor still publishes its tensor scale (amax 0 -> 1): the
  // kernel runs with one CTA and no blocks.  (An empty matrix has no scale
  // bytes, blocked or not, so nothing is left to pad.)
  if (nb == 0 && tscale_mode == FP4_TSCALE_GIVEN) return FP4_OK;
  if (dtype == FP4_BF16)
    return launch_quantize_t<true, kBlk>(x, nb, residual, rounding, seed, step, tscale_mode,
                                         tensor_scale, amax_ws, packed, scales, bm, s);
  return launch_quantize_t<false, kBlk>(x, nb, residual, rounding, seed, step, tscale_mode,
                                        tensor_scale, amax_ws, packed, scales, bm, s);
}

template <bool kG, bool kRes, bool kSR, bool kPacked>
fp4_status launch_qdq_k(uint16_t* w, const float* g, float lr, float* r, int64_t nb, uint64_t seed,
                        uint64_t step, int mode, float* ts, const float* amax, uint8_t* packed,
                        uint8_t* scales, cudaStream_t s) {
  return launch<qdq_kernel<kG, kRes, kSR, kPacked>>(nb, kThreads, 0, s, w, g, lr, r, nb, seed, step,
                                                    mode, ts, amax, packed, scales);
}

template <bool kG, bool kRes>
fp4_status launch_qdq_t(uint16_t* w, const float* g, float lr, float* r, int64_t nb, int rounding,
                        uint64_t seed, uint64_t step, int mode, float* ts, const float* amax,
                        uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  const bool pk = packed != nullptr;
  if (rounding == FP4_SR) {
    if (pk) return launch_qdq_k<kG, kRes, true, true>(w, g, lr, r, nb, seed, step, mode, ts, amax, packed, scales, s);
    return launch_qdq_k<kG, kRes, true, false>(w, g, lr, r, nb, seed, step, mode, ts, amax, packed, scales, s);
  }
  if (pk) return launch_qdq_k<kG, kRes, false, true>(w, g, lr, r, nb, seed, step, mode, ts, amax, packed, scales, s);
  return launch_qdq_k<kG, kRes, false, false>(w, g, lr, r, nb, seed, step, mode, ts, amax, packed, scales, s);
}

fp4_status launch_qdq_amax(const uint16_t* w, const float* g, float lr, const float* r, int64_t n,
                           float* amax_ws, cudaStream_t s) {
  if (cudaMemsetAsync(amax_ws, 0, sizeof(float), s) != cudaSuccess) return FP4_ERR_CUDA;
  const int64_t nb = n / 16;
  if (nb == 0) return FP4_OK;
  if (g) {
    if (r) return launch<qdq_amax_kernel<true, true>>(nb, kThreads, 0, s, w, g, lr, r, nb, amax_ws);
    return launch<qdq_amax_kernel<true, false>>(nb, kThreads, 0, s, w, g, lr, r, nb, amax_ws);
  }
  if (r) return launch<qdq_amax_kernel<false, true>>(nb, kThreads, 0, s, w, g, lr, r, nb, amax_ws);
  return launch<qdq_amax_kernel<false, false>>(nb, kThreads, 0, s, w, g, lr, r, nb, amax_ws);
}

bool mode_ok(int m) {
  return m == FP4_TSCALE_GIVEN || m == FP4_TSCALE_COMPUTE || m == FP4_TSCALE_FROM_AMAX;
}

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

fp4_status nvfp4_amax(const void* x, int dtype, int64_t n, const float* residual, float* amax_ws,
                      void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!amax_ws || (n > 0 && !x)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(residual, 32) || !aligned(amax_ws, 4)) return FP4_ERR_ALIGN;
  return launch_amax(x, dtype, n, residual, amax_ws, as_stream(stream));
}

fp4_status nvfp4_quantize(const void* x, int dtype, int64_t n, float* residual, int rounding,
                          uint64_t seed, uint64_t step, int tscale_mode, float* tensor_scale,
                          float* amax_ws, uint8_t* packed, uint8_t* scales, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (rounding != FP4_RTN && rounding != FP4_SR) return FP4_ERR_ARG;
  if (!mode_ok(tscale_mode)) return FP4_ERR_ARG;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!tensor_scale) return FP4_ERR_NULL;
  if (tscale_mode != FP4_TSCALE_GIVEN && !amax_ws) return FP4_ERR_NULL;
  if (n > 0 && (!x || !packed || !scales)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(residual, 32) || !aligned(packed, 16) ||
      !aligned(tensor_scale, 4) || !aligned(amax_ws, 4))
    return FP4_ERR_ALIGN;
  return quantize_common<false>(x, dtype, n, residual, rounding, seed, step, tscale_mode,
                                tensor_scale, amax_ws, packed, scales, BlockedMap{0, 0, 0},
                                as_stream(stream));
}

fp4_status nvfp4_quantize_blocked(const void* x, int dtype, int64_t rows, int64_t k,
                                  float* residual, int rounding, uint64_t seed, uint64_t step,
                                  int tscale_mode, float* tensor_scale, float* amax_ws,
                                  uint8_t* packed, uint8_t* blocked_scales, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (rounding != FP4_RTN && rounding != FP4_SR) return FP4_ERR_ARG;
  if (!mode_ok(tscale_mode)) return FP4_ERR_ARG;
  if (rows < 0 || k < 0 || k % 16 != 0 || k / 16 >= (INT64_C(1) << 24)) return FP4_ERR_SHAPE;
  if (k > 0 && rows > (INT64_C(1) << 44) / k) return FP4_ERR_SHAPE;
  const int64_t n = rows * k;
  if (!tensor_scale) return FP4_ERR_NULL;
  if (tscale_mode != FP4_TSCALE_GIVEN && !amax_ws) return FP4_ERR_NULL;
  if (n > 0 && (!x || !packed || !blocked_scales)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(residual, 32) || !aligned(packed, 16) ||
      !aligned(tensor_scale, 4) || !aligned(amax_ws, 4))
    return FP4_ERR_ALIGN;
  const BlockedMap bm{rows, k / 16, (k / 16 + 3) / 4};
  return quantize_common<true>(x, dtype, n, residual, rounding, seed, step, tscale_mode,
                               tensor_scale, amax_ws, packed, blocked_scales, bm,
                               as_stream(stream));
}

fp4_status nvfp4_dequantize(const uint8_t* packed, const uint8_t* scales, const float* tensor_scale,
                            int64_t n, void* y, int out_dtype, void* stream) {
  if (!dtype_ok(out_dtype)) return FP4_ERR_DTYPE;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (n > 0 && (!packed || !scales || !y)) return FP4_ERR_NULL;
  if (!aligned(packed, 16) || !aligned(scales, 2) || !aligned(y, 32) || !aligned(tensor_scale, 4))
    return FP4_ERR_ALIGN;
  const int64_t nb = n / 16;
  if (nb == 0) return FP4_OK;
  cudaStream_t s = as_stream(stream);
  const int64_t units = (nb / 2 + 1) / 2 + 1;
  if (out_dtype == FP4_BF16)
    return launch<dequantize_kernel<true>>(units, kThreads, 0, s, packed, scales, tensor_scale, nb, y);
  return launch<dequantize_kernel<false>>(units, kThreads, 0, s, packed, scales, tensor_scale, nb, y);
}

fp4_status nvfp4_qdq_amax(const uint16_t* w_bf16, const float* g, float lr, const float* residual,
                          int64_t n, float* amax_ws, void* stream) {
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!amax_ws || (n > 0 && !w_bf16)) return FP4_ERR_NULL;
  if (!aligned(w_bf16, 32) || !aligned(g, 32) || !aligned(residual, 32) || !aligned(amax_ws, 4))
    return FP4_ERR_ALIGN;
  return launch_qdq_amax(w_bf16, g, lr, residual, n, amax_ws, as_stream(stream));
}

fp4_status nvfp4_qdq(uint16_t* w_bf16, const float* g, float lr, int64_t n, float* residual,
                     int rounding, uint64_t seed, uint64_t step, int tscale_mode,
                     float* tensor_scale, float* amax_ws, uint8_t* packed, uint8_t* scales,
                     void* stream) {
  if (rounding != FP4_RTN && rounding != FP4_SR) return FP4_ERR_ARG;
  if (!mode_ok(tscale_mode)) return FP4_ERR_ARG;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!tensor_scale) return FP4_ERR_NULL;
  if (tscale_mode != FP4_TSCALE_GIVEN && !amax_ws) return FP4_ERR_NULL;
  if ((packed == nullptr) != (scales == nullptr)) return FP4_ERR_NULL;
  if (n > 0 && !w_bf16) return FP4_ERR_NULL;
  if (!aligned(w_bf16, 32) || !aligned(g, 32) || !aligned(residual, 32) || !aligned(packed, 16) ||
      !aligned(tensor_scale, 4) || !aligned(amax_ws, 4))
    return FP4_ERR_ALIGN;
  cudaStream_t s = as_stream(stream);
  if (tscale_mode == FP4_TSCALE_COMPUTE) {
    fp4_status st = launch_qdq_amax(w_bf16, g, lr, residual, n, amax_ws, s);
    if (st != FP4_OK) return st;
  }
  const int64_t nb = n / 16;
  if (nb == 0 && tscale_mode == FP4_TSCALE_GIVEN) return FP4_OK;
  if (g) {
    if (residual)
      return launch_qdq_t<true, true>(w_bf16, g, lr, residual, nb, rounding, seed, step, tscale_mode,
                                      tensor_scale, amax_ws, packed, scales, s);
    return launch_qdq_t<true, false>(w_bf16, g, lr, residual, nb, rounding, seed, step, tscale_mode,
                                     tensor_scale, amax_ws, packed, scales, s);
  }
  if (residual)
    return launch_qdq_t<false, true>(w_bf16, g, lr, residual, nb, rounding, seed, step, tscale_mode,
                                     tensor_scale, amax_ws, packed, scales, s);
  return launch_qdq_t<false, false>(w_bf16, g, lr, residual, nb, rounding, seed, step, tscale_mode,
                                    tensor_scale, amax_ws, packed, scales, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation variant of nvfp4_quantize in COMPUTE mode.
//
// The tensor-amax pass needs one fp32 of device workspace that nvfp4_quantize
// takes from its caller (amax_ws).  Some callers cannot hand one over: a
// plugin that receives only the tensors it works on from a host framework or
// inference engine that owns all device memory, or C code with no device
// allocator of its own.  For them the workspace lives in a file-scope device
// array below, which every GPU that loads this library holds until the
// process exits.

namespace fp4 {
namespace {

// 256 bytes; a call uses one fp32 slot, the tensor amax, whatever n is.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
float* g_noalloc_addr[kNoAllocMaxDevices];  // device address of the array, per device

// The array's device address on the current device.  In host code the name
// g_noalloc_scratch is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress once per device, with that device current.
fp4_status noalloc_scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return FP4_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FP4_ERR_CUDA;
    g_noalloc_addr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_addr[dev];
  return FP4_OK;
}

}  // namespace
}  // namespace fp4

extern "C" fp4_status nvfp4_quantize_noalloc(const void* x, int dtype, int64_t n, float* residual,
                                             int rounding, uint64_t seed, uint64_t step,
                                             float* tensor_scale, uint8_t* packed, uint8_t* scales,
                                             void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (rounding != FP4_RTN && rounding != FP4_SR) return FP4_ERR_ARG;
  if (n < 0 || n % 16 != 0) return FP4_ERR_SHAPE;
  if (!tensor_scale) return FP4_ERR_NULL;
  if (n > 0 && (!x || !packed || !scales)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(residual, 32) || !aligned(packed, 16) ||
      !aligned(tensor_scale, 4))
    return FP4_ERR_ALIGN;
  // Scratch this call needs: the amax slot.  It does not grow with n, so no
  // size passes the contract above and still fails here.
  const size_t need = sizeof(float);
  if (need > kNoAllocScratchBytes) return FP4_ERR_SHAPE;
  float* amax_ws = nullptr;
  fp4_status st = noalloc_scratch_address(&amax_ws);
  if (st != FP4_OK) return st;
  cudaStream_t s = as_stream(stream);
  // launch_amax clears the slot (cudaMemsetAsync) before its max pass.
  st = launch_amax(x, dtype, n, residual, amax_ws, s);
  if (st != FP4_OK) return st;
  const int64_t nb = n / 16;
  const BlockedMap linear{0, 0, 0};
  if (dtype == FP4_BF16)
    return launch_quantize_t<true, false>(x, nb, residual, rounding, seed, step,
                                          FP4_TSCALE_COMPUTE, tensor_scale, amax_ws, packed,
                                          scales, linear, s);
  return launch_quantize_t<false, false>(x, nb, residual, rounding, seed, step, FP4_TSCALE_COMPUTE,
                                         tensor_scale, amax_ws, packed, scales, linear, s);
}
