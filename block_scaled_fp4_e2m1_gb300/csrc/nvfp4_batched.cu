// nvfp4_batched.cu -- NVFP4 amax / quantize / dequantize over a list of
// independent tensors in one launch per pass.
//
// Each tensor is cut into chunks of FP4_BATCH_CHUNK_BLOCKS (256) blocks of
// 16 elements; the chunks of all tensors form one flat index space
// (fp4_tensor_desc::chunk_start, filled on the host by fp4_batch_plan), in
// which tensor t owns blocks [256 * chunk_start[t], + n_t / 16) (the rest of
// its last chunk is a hole).
//   - amax and quantize: warp w takes one contiguous range of that space,
//     ~1/nwarps of it, and walks it tensor by tensor; inside a tensor its
//     lanes stream through the blocks exactly as the single-tensor kernels
//     do (lane l: blocks l, l + 32, ...), with their loads in flight ahead.
//     A warp meets a tensor boundary once or twice, so the per-tensor set-up
//     (locating it, its scale) costs nothing on the way.
//   - dequantize: warps take whole chunks in grid-stride order and locate
//     each chunk's tensor by a 32-way search over the descriptors.
// Either way every lane of a warp works on the same tensor, and the
// arithmetic per block is the single-tensor kernels' (nvfp4_device.cuh), so
// each tensor's result is bit-identical to the single-tensor call.
//
// This removes the per-launch ramp and tail of many small launches: a model
// of a few hundred weight matrices is one amax, one quantize and one
// dequantize launch instead of hundreds of each.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"
#include "nvfp4_device.cuh"

namespace fp4 {
namespace {

constexpr int kBThreads = 256;
constexpr int kChunk = FP4_BATCH_CHUNK_BLOCKS;
constexpr int kLaneBlocks = kChunk / 32;  // blocks per lane per chunk

__device__ __forceinline__ int64_t ldg_i64(const int64_t* p) {
  return (int64_t)__ldg(reinterpret_cast<const long long*>(p));
}

template <typename T>
__device__ __forceinline__ T* ldg_ptr(T* const* p) {
  return reinterpret_cast<T*>(__ldg(reinterpret_cast<const unsigned long long*>(p)));
}

// Largest t in [0, count) with desc[t].chunk_start <= c (chunk_start is
// non-decreasing and desc[0].chunk_start = 0 <= c): a 32-way warp search.
__device__ __forceinline__ int find_tensor(const fp4_tensor_desc* __restrict__ d, int count,
                                           int64_t c) {
  int lo = 0, hi = count;
  const int lane = threadIdx.x & 31;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool ok = idx < hi && ldg_i64(&d[idx].chunk_start) <= c;
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, ok);
    lo += (31 - __clz(ball)) * step;
    hi = lo + step < hi ? lo + step : hi;
  }
  return lo;
}

// The chunk a warp works on: its tensor and its block range.
struct Chunk {
  int t;
  int64_t b0;  // first block of the chunk inside the tensor
  int64_t nb;  // blocks of the tensor
  int64_t j;   // chunk index inside the tensor
};

__device__ __forceinline__ Chunk locate(const fp4_tensor_desc* __restrict__ desc, int count,
                                        int64_t c) {
  Chunk k;
  k.t = find_tensor(desc, count, c);
  k.j = c - ldg_i64(&desc[k.t].chunk_start);
  k.b0 = k.j * kChunk;
  k.nb = ldg_i64(&desc[k.t].n) / 16;
  return k;
}

// This warp's range [r0, r1) of the flat block space, whole warps of 32.
struct WarpRange {
  int64_t r0, r1;
};

__device__ __forceinline__ WarpRange warp_range(int64_t total_chunks) {
  const int64_t nwarps = (int64_t)gridDim.x * (kBThreads / 32);
  const int64_t w = (int64_t)blockIdx.x * (kBThreads / 32) + (threadIdx.x >> 5);
  const int64_t total = total_chunks * kChunk;
  const int64_t len = ((total + nwarps - 1) / nwarps + 31) & ~int64_t(31);
  const int64_t r0 = w * len;
  return WarpRange{r0 < total ? r0 : total, r0 + len < total ? r0 + len : total};
}

// Walks this warp's range tensor by tensor (warp-uniform): seg(t, s0, s1)
// gets the blocks [s0, s1) of tensor t that fall into the range.
template <typename Seg>
__device__ __forceinline__ void for_each_segment(const fp4_tensor_desc* __restrict__ desc,
                                                 int count, int64_t total_chunks, Seg seg) {
  const WarpRange wr = warp_range(total_chunks);
  if (wr.r0 >= wr.r1) return;
  int64_t r0 = wr.r0;
  for (int t = find_tensor(desc, count, r0 / kChunk); t < count && r0 < wr.r1; ++t) {
    const int64_t tb0 = ldg_i64(&desc[t].chunk_start) * kChunk;
    const int64_t nb = ldg_i64(&desc[t].n) / 16;
    const int64_t s0 = (r0 > tb0 ? r0 : tb0) - tb0;
    const int64_t s1 = wr.r1 - tb0 < nb ? wr.r1 - tb0 : nb;
    if (s0 < s1) seg(t, s0, s1);
    if (t + 1 < count) {
      const int64_t next = ldg_i64(&desc[t + 1].chunk_start) * kChunk;
      if (next > r0) r0 = next;
    }
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kBThreads)
    amax_batched_kernel(const fp4_tensor_desc* __restrict__ desc, int count, int64_t total_chunks,
                        float* __restrict__ amax) {
  constexpr int kWords = kBF16 ? 1 : 2;
  constexpr int kU = 4;  // blocks a lane has in flight
  const int lane = threadIdx.x & 31;
  for_each_segment(desc, count, total_chunks, [&](int t, int64_t s0, int64_t s1) {
    const uint8_t* x = static_cast<const uint8_t*>(ldg_ptr(&desc[t].x));
    float m = 0.0f;
    for (int64_t b0 = s0 + lane; b0 < s1; b0 += 32 * kU) {
      U32x8 raw[kU][kWords];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t b = b0 + 32 * u;
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
          if (b < s1) {
            raw[u][w] = ld_stream_v8(x + b * (32 * kWords) + 32 * w);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) raw[u][w].w[i] = 0u;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (kBF16) {
            m = fmaxf(m, fabsf(bf16_lo(raw[u][0].w[i])));
            m = fmaxf(m, fabsf(bf16_hi(raw[u][0].w[i])));
          } else {
            m = fmaxf(m, fabsf(__uint_as_float(raw[u][0].w[i])));
            m = fmaxf(m, fabsf(__uint_as_float(raw[u][kWords - 1].w[i])));
          }
        }
    }
    const uint32_t wm = warp_max_u32(__float_as_uint(m));
    if (lane == 0 && wm != 0u) atomicMax(reinterpret_cast<unsigned int*>(amax + t), wm);
  });
}

// Inside a tensor a lane quantizes blocks s0 + lane, + 32, ... with the
// loads of its next kD blocks in flight (the single-tensor kernel's ring).
// bf16 round-to-nearest refills the warp's table of E2M1 constants for each
// tensor it enters.
template <bool kBF16, bool kSR>
__global__ void __launch_bounds__(kBThreads, kSR ? 1 : (kBF16 ? 3 : 2))
    quantize_batched_kernel(const fp4_tensor_desc* __restrict__ desc, int count,
                            int64_t total_chunks, uint64_t seed, uint64_t step, int tscale_mode,
                            float* __restrict__ tensor_scale, const float* __restrict__ amax) {
  constexpr int kD = kBF16 ? 2 : 1;  // blocks in flight ahead of the one being quantized
  constexpr bool kFast = kBF16 && !kSR;
  __shared__ EffEntry eff_tabs[kFast ? (kBThreads / 32) * kEffEntries : 1];
  EffEntry* const tab = eff_tabs + (kFast ? (threadIdx.x >> 5) * kEffEntries : 0);
  const int lane = threadIdx.x & 31;
  const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
  const uint32_t st0 = (uint32_t)step, st1 = (uint32_t)(step >> 32);
  for_each_segment(desc, count, total_chunks, [&](int t, int64_t s0, int64_t s1) {
    const float s_t = tscale_mode == FP4_TSCALE_GIVEN ? sanitize_scale(tensor_scale[t])
                                                      : tensor_scale_from_amax(amax[t]);
    if (tscale_mode != FP4_TSCALE_GIVEN && s0 == 0 && lane == 0) tensor_scale[t] = s_t;
    const ScaleDiv sd = make_scale_div(s_t);
    if (kFast) build_eff_table(tab, s_t);
    const void* x = ldg_ptr(&desc[t].x);
    uint8_t* const packed = ldg_ptr(&desc[t].packed);
    uint8_t* const scales = ldg_ptr(&desc[t].scales);
    int64_t b = s0 + lane;
    BlockIn<kBF16, false> buf[kD + 1];
#pragma unroll
    for (int d = 0; d < kD; ++d) issue_block<kBF16, false>(x, nullptr, b + 32 * d, s1, buf[d]);
    for (;;) {
#pragma unroll
      for (int r = 0; r <= kD; ++r) {
        if (b >= s1) goto segment_done;
        issue_block<kBF16, false>(x, nullptr, b + 32 * kD, s1, buf[(r + kD) % (kD + 1)]);
        uint2 out;
        uint32_t sb;
        if (kFast) {
          sb = quantize_block_bf16_rtn(buf[r].x[0], sd, tab, out);
        } else {
          float v[16], rr[16], q[16];
          unpack_block<kBF16, false>(buf[r], v, rr);
          sb = quantize_block<kSR, false>(v, s_t, sd, (uint64_t)(16 * b), key0, key1, st0, st1,
                                          out, q);
        }
        *reinterpret_cast<uint2*>(packed + 8 * b) = out;
        scales[b] = (uint8_t)sb;
        b += 32;
      }
    }
  segment_done:;
  });
}

// The blocked-scale variant walks the tensors one after the other, each
// with the whole grid in grid-stride order (the single-tensor kernel's
// order), not in per-warp ranges.  A tensor's scale tiles are then
// completed by the whole GPU within a pass or two, so their 16-byte lines
// fill in L2 at once.  With per-warp ranges, thousands of warps each kept
// their own row tiles half written, the partial lines overflowed L2, and
// the kernel ran at 0.6 of the copy bandwidth.  tensor t's scales go to the
// blocked layout of its [n_t / k_t, k_t] matrix (k: device array of the
// k_t); padding is zeroed by the whole grid.
template <bool kBF16, bool kSR>
__global__ void __launch_bounds__(kBThreads, kSR ? 1 : (kBF16 ? 3 : 2))
    quantize_batched_blocked_kernel(const fp4_tensor_desc* __restrict__ desc, int count,
                                    const int64_t* __restrict__ kdim, uint64_t seed, uint64_t step,
                                    int tscale_mode, float* __restrict__ tensor_scale,
                                    const float* __restrict__ amax) {
  constexpr int kD = kBF16 ? 2 : 1;  // blocks in flight ahead of the one being quantized
  constexpr bool kFast = kBF16 && !kSR;
  __shared__ EffEntry eff_tabs[kFast ? (kBThreads / 32) * kEffEntries : 1];
  EffEntry* const tab = eff_tabs + (kFast ? (threadIdx.x >> 5) * kEffEntries : 0);
  const uint32_t key0 = (uint32_t)seed, key1 = (uint32_t)(seed >> 32);
  const uint32_t st0 = (uint32_t)step, st1 = (uint32_t)(step >> 32);
  const int64_t stride = (int64_t)gridDim.x * kBThreads;
  const int64_t gtid = (int64_t)blockIdx.x * kBThreads + threadIdx.x;
  for (int t = 0; t < count; ++t) {
    const float s_t = tscale_mode == FP4_TSCALE_GIVEN ? sanitize_scale(tensor_scale[t])
                                                      : tensor_scale_from_amax(amax[t]);
    if (tscale_mode != FP4_TSCALE_GIVEN && gtid == 0) tensor_scale[t] = s_t;
    const int64_t nb = ldg_i64(&desc[t].n) / 16;
    if (nb == 0) continue;
    const ScaleDiv sd = make_scale_div(s_t);
    if (kFast) build_eff_table(tab, s_t);
    const void* x = ldg_ptr(&desc[t].x);
    uint8_t* const packed = ldg_ptr(&desc[t].packed);
    uint8_t* const scales = ldg_ptr(&desc[t].scales);
    const int64_t kc = ldg_i64(&kdim[t]) / 16;  // block scales per row
    const BlockedMap bm{nb / kc, kc, (kc + 3) / 4};
    blocked_zero_padding(scales, bm.rows, bm.cols, bm.col_tiles, gtid, stride);
    int64_t b = gtid;
    BlockedCursor cur = blocked_cursor(b, bm);
    const BlockedStep cstep = blocked_step(stride, bm);
    BlockIn<kBF16, false> buf[kD + 1];
#pragma unroll
    for (int d = 0; d < kD; ++d) issue_block<kBF16, false>(x, nullptr, b + d * stride, nb, buf[d]);
    for (;;) {
#pragma unroll
      for (int r = 0; r <= kD; ++r) {
        if (b >= nb) goto tensor_done;
        issue_block<kBF16, false>(x, nullptr, b + kD * stride, nb, buf[(r + kD) % (kD + 1)]);
        uint2 out;
        uint32_t sb;
        if (kFast) {
          sb = quantize_block_bf16_rtn(buf[r].x[0], sd, tab, out);
        } else {
          float v[16], rr[16], q[16];
          unpack_block<kBF16, false>(buf[r], v, rr);
          sb = quantize_block<kSR, false>(v, s_t, sd, (uint64_t)(16 * b), key0, key1, st0, st1,
                                          out, q);
        }
        *reinterpret_cast<uint2*>(packed + 8 * b) = out;
        scales[blocked_at(cur)] = (uint8_t)sb;
        blocked_advance(cur, cstep);
        b += stride;
      }
    }
  tensor_done:;
  }
}

template <bool kBF16Out>
__global__ void __launch_bounds__(kBThreads)
    dequantize_batched_kernel(const fp4_tensor_desc* __restrict__ desc, int count,
                              int64_t total_chunks, const float* __restrict__ tensor_scale) {
  constexpr int kLanePairs = kLaneBlocks / 2;  // two-block units per lane per chunk
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (kBThreads / 32);
  int cur_t = -1;
  float s_t = 1.0f;
  for (int64_t c = (int64_t)blockIdx.x * (kBThreads / 32) + (threadIdx.x >> 5); c < total_chunks;
       c += nwarps) {
    const Chunk k = locate(desc, count, c);
    if (k.t != cur_t) {
      cur_t = k.t;
      s_t = tensor_scale ? sanitize_scale(tensor_scale[k.t]) : 1.0f;
    }
    const uint8_t* packed = ldg_ptr(&desc[k.t].packed);
    const uint8_t* scales = ldg_ptr(&desc[k.t].scales);
    void* y = ldg_ptr(&desc[k.t].y);
    uint4 pk[kLanePairs];
    uint32_t sc[kLanePairs];
#pragma unroll
    for (int u = 0; u < kLanePairs; ++u) {
      const int64_t b = k.b0 + 2 * (lane + 32 * u);  // first block of the pair
      if (b + 1 < k.nb) {
        pk[u] = ld_stream_v4(packed + 8 * b);
        uint16_t s2;
        asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(s2) : "l"(scales + b));
        sc[u] = s2;
      } else if (b < k.nb) {  // the odd last block of a tensor
        const uint2 q = ld_stream_v2(packed + 8 * b);
        pk[u] = make_uint4(q.x, q.y, 0u, 0u);
        sc[u] = ld_stream_u8(scales + b);
      }
    }
#pragma unroll
    for (int u = 0; u < kLanePairs; ++u) {
      const int64_t b = k.b0 + 2 * (lane + 32 * u);
      if (b < k.nb)
        dequantize_store<kBF16Out>(pk[u].x, pk[u].y, __fmul_rn(e4m3_value(sc[u] & 0xFFu), s_t), y,
                                   b);
      if (b + 1 < k.nb)
        dequantize_store<kBF16Out>(pk[u].z, pk[u].w, __fmul_rn(e4m3_value(sc[u] >> 8), s_t), y,
                                   b + 1);
    }
  }
}

fp4_status check_desc(const fp4_tensor_desc* desc, int32_t count, int64_t total_chunks) {
  if (count < 0 || count >= (1 << 24) || total_chunks < 0) return FP4_ERR_SHAPE;
  if (count > 0 && desc == nullptr) return FP4_ERR_NULL;
  if (!aligned(desc, 8)) return FP4_ERR_ALIGN;
  return FP4_OK;
}

fp4_status launch_amax_batched(const fp4_tensor_desc* desc, int32_t count, int64_t total_chunks,
                               int dtype, float* amax, cudaStream_t s) {
  if (count > 0 && cudaMemsetAsync(amax, 0, sizeof(float) * (size_t)count, s) != cudaSuccess)
    return FP4_ERR_CUDA;
  if (total_chunks == 0) return FP4_OK;
  if (dtype == FP4_BF16)
    return launch<amax_batched_kernel<true>>(total_chunks * kChunk, kBThreads, 0, s, desc, count,
                                             total_chunks, amax);
  return launch<amax_batched_kernel<false>>(total_chunks * kChunk, kBThreads, 0, s, desc, count,
                                            total_chunks, amax);
}

template <bool kBlk>
fp4_status quantize_batched_common(const fp4_tensor_desc* desc, const int64_t* k, int32_t count,
                                   int64_t total_chunks, int dtype, int rounding, uint64_t seed,
                                   uint64_t step, int tscale_mode, float* tensor_scale,
                                   float* amax, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (rounding != FP4_RTN && rounding != FP4_SR) return FP4_ERR_ARG;
  if (tscale_mode != FP4_TSCALE_GIVEN && tscale_mode != FP4_TSCALE_COMPUTE &&
      tscale_mode != FP4_TSCALE_FROM_AMAX)
    return FP4_ERR_ARG;
  if (const fp4_status st = check_desc(desc, count, total_chunks); st != FP4_OK) return st;
  if (count > 0 && !tensor_scale) return FP4_ERR_NULL;
  if (count > 0 && tscale_mode != FP4_TSCALE_GIVEN && !amax) return FP4_ERR_NULL;
  if (!aligned(tensor_scale, 4) || !aligned(amax, 4)) return FP4_ERR_ALIGN;
  cudaStream_t s = as_stream(stream);
  if (tscale_mode == FP4_TSCALE_COMPUTE) {
    const fp4_status st = launch_amax_batched(desc, count, total_chunks, dtype, amax, s);
    if (st != FP4_OK) return st;
  }
  if (total_chunks == 0) return FP4_OK;
  const int64_t units = total_chunks * kChunk;  // one thread per block of the flat space
  if (kBlk) {
    if (dtype == FP4_BF16) {
      if (rounding == FP4_SR)
        return launch<quantize_batched_blocked_kernel<true, true>>(
            units, kBThreads, 0, s, desc, count, k, seed, step, tscale_mode, tensor_scale, amax);
      return launch<quantize_batched_blocked_kernel<true, false>>(
          units, kBThreads, 0, s, desc, count, k, seed, step, tscale_mode, tensor_scale, amax);
    }
    if (rounding == FP4_SR)
      return launch<quantize_batched_blocked_kernel<false, true>>(
          units, kBThreads, 0, s, desc, count, k, seed, step, tscale_mode, tensor_scale, amax);
    return launch<quantize_batched_blocked_kernel<false, false>>(
        units, kBThreads, 0, s, desc, count, k, seed, step, tscale_mode, tensor_scale, amax);
  }
  if (dtype == FP4_BF16) {
    if (rounding == FP4_SR)
      return launch<quantize_batched_kernel<true, true>>(units, kBThreads, 0, s, desc, count,
                                                         total_chunks, seed, step, tscale_mode,
                                                         tensor_scale, amax);
    return launch<quantize_batched_kernel<true, false>>(units, kBThreads, 0, s, desc, count,
                                                        total_chunks, seed, step, tscale_mode,
                                                        tensor_scale, amax);
  }
  if (rounding == FP4_SR)
    return launch<quantize_batched_kernel<false, true>>(units, kBThreads, 0, s, desc, count,
                                                        total_chunks, seed, step, tscale_mode,
                                                        tensor_scale, amax);
  return launch<quantize_batched_kernel<false, false>>(units, kBThreads, 0, s, desc, count,
                                                       total_chunks, seed, step, tscale_mode,
                                                       tensor_scale, amax);
}

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

fp4_status fp4_batch_plan(fp4_tensor_desc* host_desc, int32_t count, int64_t* total_chunks) {
  if (!total_chunks || (count > 0 && !host_desc)) return FP4_ERR_NULL;
  if (count < 0 || count >= (1 << 24)) return FP4_ERR_SHAPE;
  for (int32_t t = 0; t < count; ++t) {
    const fp4_tensor_desc& d = host_desc[t];
    if (d.n < 0 || d.n % 16 != 0 || d.n >= (int64_t(16) << 40)) return FP4_ERR_SHAPE;
    if (!aligned(d.x, 32) || !aligned(d.packed, 16) || !aligned(d.scales, 2) || !aligned(d.y, 32))
      return FP4_ERR_ALIGN;
  }
  int64_t acc = 0;
  for (int32_t t = 0; t < count; ++t) {
    host_desc[t].chunk_start = acc;
    acc += (host_desc[t].n / 16 + kChunk - 1) / kChunk;
  }
  *total_chunks = acc;
  return FP4_OK;
}

fp4_status nvfp4_amax_batched(const fp4_tensor_desc* desc, int32_t count, int64_t total_chunks,
                              int dtype, float* amax, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (const fp4_status st = check_desc(desc, count, total_chunks); st != FP4_OK) return st;
  if (count > 0 && !amax) return FP4_ERR_NULL;
  if (!aligned(amax, 4)) return FP4_ERR_ALIGN;
  return launch_amax_batched(desc, count, total_chunks, dtype, amax, as_stream(stream));
}

fp4_status nvfp4_quantize_batched(const fp4_tensor_desc* desc, int32_t count, int64_t total_chunks,
                                  int dtype, int rounding, uint64_t seed, uint64_t step,
                                  int tscale_mode, float* tensor_scale, float* amax, void* stream) {
  return quantize_batched_common<false>(desc, nullptr, count, total_chunks, dtype, rounding, seed,
                                        step, tscale_mode, tensor_scale, amax, stream);
}

fp4_status nvfp4_quantize_batched_blocked(const fp4_tensor_desc* desc, const int64_t* k,
                                          int32_t count, int64_t total_chunks, int dtype,
                                          int rounding, uint64_t seed, uint64_t step,
                                          int tscale_mode, float* tensor_scale, float* amax,
                                          void* stream) {
  if (count > 0 && !k) return FP4_ERR_NULL;
  if (!aligned(k, 8)) return FP4_ERR_ALIGN;
  return quantize_batched_common<true>(desc, k, count, total_chunks, dtype, rounding, seed, step,
                                       tscale_mode, tensor_scale, amax, stream);
}

fp4_status fp4_batch_plan_blocked(fp4_tensor_desc* host_desc, const int64_t* host_k, int32_t count,
                                  int64_t* total_chunks) {
  if (count > 0 && !host_k) return FP4_ERR_NULL;
  for (int32_t t = 0; t < count && host_desc; ++t) {
    const int64_t k = host_k[t], n = host_desc[t].n;
    if (k <= 0 || k % 16 != 0 || k / 16 >= (INT64_C(1) << 24) || n % k != 0) return FP4_ERR_SHAPE;
  }
  return fp4_batch_plan(host_desc, count, total_chunks);
}

fp4_status nvfp4_dequantize_batched(const fp4_tensor_desc* desc, int32_t count,
                                    int64_t total_chunks, const float* tensor_scale, int out_dtype,
                                    void* stream) {
  if (!dtype_ok(out_dtype)) return FP4_ERR_DTYPE;
  if (const fp4_status st = check_desc(desc, count, total_chunks); st != FP4_OK) return st;
  if (!aligned(tensor_scale, 4)) return FP4_ERR_ALIGN;
  if (total_chunks == 0) return FP4_OK;
  const int64_t units = total_chunks * 32;
  cudaStream_t s = as_stream(stream);
  if (out_dtype == FP4_BF16)
    return launch<dequantize_batched_kernel<true>>(units, kBThreads, 0, s, desc, count,
                                                   total_chunks, tensor_scale);
  return launch<dequantize_batched_kernel<false>>(units, kBThreads, 0, s, desc, count,
                                                  total_chunks, tensor_scale);
}

}  // extern "C"
