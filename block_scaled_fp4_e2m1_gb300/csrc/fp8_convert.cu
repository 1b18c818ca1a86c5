// fp8_convert.cu -- direct MXFP4 -> FP8 E4M3 conversion, row form
// (FP4RowToFP8Row) and fused transposed column form over ragged expert
// segments (FP4RowToFP8Col).
//
// [MoE-FP4] "核心技术贡献" 1: the E2M1 exponent is re-biased into E4M3
// (E_fp8 = E_fp4 - 1 + 7), the mantissa bit shifts into the E4M3 mantissa
// field, and four 32-element MXFP4 blocks share one 128-element FP8 block
// whose scale S_t is the largest of their UE8M0 scales, each element's
// exponent lowered by S_t - S_sub; all by bit operations, no math library.
// Defined result: the E4M3 value nearest to value(code) * 2^-(S_t - S_sub)
// (exact unless S_t - S_sub >= 9); fp32 output scale 2^(S_t - 127).
//
// Bit mapping: for a shift d the 8 magnitudes of E2M1 map to 8 E4M3 bytes,
// a table of 8 bytes held in two 32-bit words.  A packed word of 8 codes
// becomes 8 E4M3 bytes with two byte permutes (prmt) that look the
// magnitudes up in that table, two more that replicate each code's sign bit
// into a byte mask, and two 3-input logic ops that merge them.  The 16
// tables (d >= 13 is all zero; d is clamped to 15) are built once per CTA in
// shared memory with the hardware round-to-nearest E4M3 conversion of the
// exact values value(j) * 2^-d.
//
// [MoE-FP4] "核心技术贡献" 2 and 3: FP4RowToFP8Col fuses dequantize,
// transpose and requantize in one pass (the page stages the transpose
// through a padded shared-memory tile; here each warp transposes its block
// in registers, see the column kernel), over ragged per-expert row segments
// located by precomputed offsets.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"

namespace fp4 {
namespace {

// 16 tables of 8 bytes: table d holds E4M3(value(j) * 2^-d), j = 0..7.
__device__ __forceinline__ void build_shift_tables(uint8_t* lut) {
  const int t = threadIdx.x;
  if (t < 128) {
    const int d = t >> 3, j = t & 7;
    const float scale = __uint_as_float((uint32_t)(127 - d) << 23);  // 2^-d
    lut[t] = (uint8_t)cvt_e4m3(__fmul_rn(e2m1_value((uint32_t)j), scale));
  }
}

// prmt.b32 in its generic mode: each selector nibble picks one of the 8
// bytes of {b, a} with bits 2:0 and, when bit 3 is set, replicates that
// byte's bit 7 over the whole byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// 8 codes (w, code i in bits 4i+3..4i) -> 8 E4M3 bytes (lo: codes 0-3).
__device__ __forceinline__ void convert8(uint32_t w, uint2 lut, uint32_t& lo, uint32_t& hi) {
  const uint32_t mag = w & 0x77777777u;
  const uint32_t even_sign = w << 4;  // byte k bit 7 = sign of code 2k
  const uint32_t m_lo = prmt(lut.x, lut.y, mag);
  const uint32_t m_hi = prmt(lut.x, lut.y, mag >> 16);
  // selector nibbles with bit 3 set replicate the chosen byte's bit 7
  const uint32_t s_lo = prmt(even_sign, w, 0xD9C8u);  // signs of codes 0,1,2,3
  const uint32_t s_hi = prmt(even_sign, w, 0xFBEAu);  // signs of codes 4,5,6,7
  lo = m_lo | (s_lo & 0x80808080u);
  hi = m_hi | (s_hi & 0x80808080u);
}

__device__ __forceinline__ uint32_t max_byte4(uint32_t s) {
  uint32_t m = __vmaxu4(s, s >> 16);
  m = __vmaxu4(m, m >> 8);
  return m & 0xFFu;
}

// fp32 2^(S - 127) for a UE8M0 byte S (S = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t s) {
  return __uint_as_float(s == 0u ? 0x00400000u : (s << 23));
}

// ------------------------------------------------------------------- row

constexpr int kRowThreads = 256;

// One thread per 128-element span: 64 B of codes, 4 scale bytes in; 128 B of
// E4M3 and one fp32 scale out.  Spans of all rows are contiguous in flat
// order because cols % 128 == 0.
__global__ void __launch_bounds__(kRowThreads)
    fp4_to_fp8_row_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                          int64_t nspans, uint8_t* __restrict__ fp8, float* __restrict__ fp8_scales) {
  __shared__ __align__(8) uint8_t lut[128];
  build_shift_tables(lut);
  __syncthreads();
  const uint2* lut2 = reinterpret_cast<const uint2*>(lut);
  const int64_t stride = (int64_t)gridDim.x * kRowThreads;
  for (int64_t j = (int64_t)blockIdx.x * kRowThreads + threadIdx.x; j < nspans; j += stride) {
    const uint32_t sc = ld_stream_u32(scales + 4 * j);
    const U32x8 p0 = ld_stream_v8(packed + 64 * j);
    const U32x8 p1 = ld_stream_v8(packed + 64 * j + 32);
    const uint32_t st = max_byte4(sc);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t d = st - ((sc >> (8 * k)) & 0xFFu);
      d = d > 15u ? 15u : d;
      const uint2 l = lut2[d];
      U32x8 o;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w = (k < 2) ? p0.w[4 * k + i] : p1.w[4 * (k - 2) + i];
        convert8(w, l, o.w[2 * i], o.w[2 * i + 1]);
      }
      st_v8(fp8 + 128 * j + 32 * k, o);
    }
    fp8_scales[j] = ue8m0_to_f32(st);
  }
}

// ------------------------------------------------------------------- col
//
// Work unit: one warp converts one FP8 scale block, i.e. 128 tokens of one
// segment x 32 features (one MXFP4 scale column).  Lane (g, c) = (lane & 7,
// lane >> 3) owns tokens 16g .. 16g+15 and features 8c .. 8c+7 of the unit:
// it loads one 32-bit word of 8 codes and one scale byte per token, the warp
// reduces the block's target scale with three shuffles, each lane converts
// its 16 words through the shift tables and transposes them into 8 feature
// rows x 16 token bytes, and writes those rows to the (unaligned) segment
// output with aligned 16-byte stores assembled from its own bytes and the
// next lane's.  No shared-memory tile and no CTA barrier: the warps of a
// CTA are independent, and consecutive warps take neighbouring feature
// blocks of the same token block so their 16-byte row slices share sectors.

constexpr int kColThreads = 256;

// Largest e in [0, nseg) with off[e] <= v, for off non-decreasing, off[0] = 0
// <= v < off[nseg]: a 32-way search by one warp.
__device__ __forceinline__ int find_segment(const int64_t* __restrict__ off, int nseg, int64_t v) {
  int lo = 0, hi = nseg;  // answer in [lo, hi)
  const int lane = threadIdx.x & 31;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool ok = idx < hi && off[idx] <= v;
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, ok);
    const int last = 31 - __clz(ball);  // lane 0 is always true
    lo = lo + last * step;
    const int nhi = lo + step;
    hi = nhi < hi ? nhi : hi;
  }
  return lo;
}

// Bytes o .. o+15 (1 <= o <= 15) of the 32-byte sequence x[0..3] | y[0..3].
__device__ __forceinline__ uint4 window16(uint4 x, uint4 y, int o) {
  uint32_t w0 = x.x, w1 = x.y, w2 = x.z, w3 = x.w, w4 = y.x, w5 = y.y, w6 = y.z, w7 = y.w;
  if (o & 8) {
    w0 = w2; w1 = w3; w2 = w4; w3 = w5; w4 = w6; w5 = w7;
  }
  if (o & 4) {
    w0 = w1; w1 = w2; w2 = w3; w3 = w4; w4 = w5;
  }
  const uint32_t sh = 8u * (uint32_t)(o & 3);
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                    __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// Store bytes lo .. hi-1 (0 <= lo < hi <= 16) of the 16-byte value v to the
// 16-byte aligned p: one 128-bit store when the chunk is whole, otherwise
// the whole 32-bit words inside [lo, hi) as word stores and the bytes of the
// (at most two) edge words as byte stores, all predicated, no loop.
__device__ __forceinline__ void store_chunk(uint8_t* p, uint4 v, int lo, int hi) {
  if (lo <= 0 && hi >= 16) {
    *reinterpret_cast<uint4*>(p) = v;
    return;
  }
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (lo <= 4 * t && 4 * t + 4 <= hi) reinterpret_cast<uint32_t*>(p)[t] = vw[t];
  // edge words: the word holding byte lo (if lo is not word aligned) and the
  // word holding byte hi - 1 (if hi is not word aligned)
  const int wl = lo >> 2, wh = (hi - 1) >> 2;
  const uint32_t xl = vw[0] * (wl == 0) + vw[1] * (wl == 1) + vw[2] * (wl == 2) + vw[3] * (wl == 3);
  const uint32_t xh = vw[0] * (wh == 0) + vw[1] * (wh == 1) + vw[2] * (wh == 2) + vw[3] * (wh == 3);
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    if ((lo & 3) != 0 && q < 4 - (lo & 3) && lo + q < hi)
      p[lo + q] = (uint8_t)(xl >> (8 * ((lo + q) & 3)));
    const int bh = 4 * wh + q;      // bytes of the last word before hi
    if ((hi & 3) != 0 && q < (hi & 3) && bh >= lo && (wl != wh || (lo & 3) == 0))
      p[bh] = (uint8_t)(xh >> (8 * q));
  }
}

__global__ void __launch_bounds__(kColThreads)
    fp4_to_fp8_col_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                          int64_t cols, const int64_t* __restrict__ seg_row_off,
                          const int64_t* __restrict__ seg_scale_off, int nseg, int64_t nunits,
                          uint8_t* __restrict__ fp8_t, float* __restrict__ fp8_t_scales) {
  __shared__ __align__(8) uint8_t lut[128];
  build_shift_tables(lut);
  __syncthreads();
  const uint2* lut2 = reinterpret_cast<const uint2*>(lut);
  const int lane = threadIdx.x & 31;
  const int g = lane & 7;   // token group
  const int c = lane >> 3;  // 8-feature slice of the 32-feature block
  const int64_t kblocks = cols / 32;
  const int64_t row_bytes = cols / 2;
  const int64_t nwarps = (int64_t)gridDim.x * (kColThreads / 32);
  for (int64_t unit = (int64_t)blockIdx.x * (kColThreads / 32) + (threadIdx.x >> 5); unit < nunits;
       unit += nwarps) {
    const int64_t fb = unit / kblocks;              // global token block
    const int kb = (int)(unit - fb * kblocks);      // feature block
    const int e = find_segment(seg_scale_off, nseg, fb);
    const int64_t row0 = seg_row_off[e];
    const int64_t n_e = seg_row_off[e + 1] - row0;
    const int64_t sofs = seg_scale_off[e];
    const int64_t b = fb - sofs;
    const int64_t left = n_e - 128 * b;
    const int nv = left < 128 ? (int)left : 128;    // tokens in this block

    // Load: 16 tokens x (8 codes, 1 scale byte).
    uint32_t w[16], s[16];
    {
      const int64_t r = row0 + 128 * b + 16 * g;
      const uint8_t* pw = packed + r * row_bytes + 16 * kb + 4 * c;
      const uint8_t* ps = scales + r * kblocks + kb;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool ok = 16 * g + i < nv;
        w[i] = ok ? ld_stream_u32(pw + i * row_bytes) : 0u;
        s[i] = ok ? ld_stream_u8(ps + i * kblocks) : 0u;
      }
    }
    // Target scale: the block's largest source scale.
    uint32_t st = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) st = max(st, s[i]);
    st = max(st, __shfl_xor_sync(0xFFFFFFFFu, st, 1));
    st = max(st, __shfl_xor_sync(0xFFFFFFFFu, st, 2));
    st = max(st, __shfl_xor_sync(0xFFFFFFFFu, st, 4));
    const int64_t nb_e = (n_e + 127) / 128;
    fp8_t_scales[cols * sofs + (32 * kb + lane) * nb_e + b] = ue8m0_to_f32(st);

    // Convert and transpose: o[f][q] = 4 token bytes (16g + 4q ..) of feature 8c + f.
    uint32_t o[8][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t d = st - s[4 * q + i];
        d = d > 15u ? 15u : d;
        convert8(w[4 * q + i], lut2[d], lo[i], hi[i]);
      }
      const uint32_t a0 = __byte_perm(lo[0], lo[1], 0x5140u), a1 = __byte_perm(lo[0], lo[1], 0x7362u);
      const uint32_t a2 = __byte_perm(lo[2], lo[3], 0x5140u), a3 = __byte_perm(lo[2], lo[3], 0x7362u);
      const uint32_t b0 = __byte_perm(hi[0], hi[1], 0x5140u), b1 = __byte_perm(hi[0], hi[1], 0x7362u);
      const uint32_t b2 = __byte_perm(hi[2], hi[3], 0x5140u), b3 = __byte_perm(hi[2], hi[3], 0x7362u);
      o[0][q] = __byte_perm(a0, a2, 0x5410u);
      o[1][q] = __byte_perm(a0, a2, 0x7632u);
      o[2][q] = __byte_perm(a1, a3, 0x5410u);
      o[3][q] = __byte_perm(a1, a3, 0x7632u);
      o[4][q] = __byte_perm(b0, b2, 0x5410u);
      o[5][q] = __byte_perm(b0, b2, 0x7632u);
      o[6][q] = __byte_perm(b1, b3, 0x5410u);
      o[7][q] = __byte_perm(b1, b3, 0x7632u);
    }

    // Store: feature row k = 32kb + 8c + f holds the block's nv tokens at
    // S = fp8_t + cols*row0 + k*n_e + 128b, a = S mod 16.  With a = 0 lane g
    // writes bytes 16g .. 16g+15 as they are; otherwise it writes the
    // aligned chunk starting at token 16g + 16 - a (its last a bytes and the
    // next lane's first 16 - a bytes), and lane 0 also the head chunk.
    uint8_t* const blk = fp8_t + cols * row0 + 128 * b;
    const int own_end = nv - 16 * g;  // bytes of this lane's 16 that are valid (may be <= 0)
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      const uint4 mine = make_uint4(o[f][0], o[f][1], o[f][2], o[f][3]);
      const uint4 next = make_uint4(__shfl_down_sync(0xFFFFFFFFu, mine.x, 1),
                                    __shfl_down_sync(0xFFFFFFFFu, mine.y, 1),
                                    __shfl_down_sync(0xFFFFFFFFu, mine.z, 1),
                                    __shfl_down_sync(0xFFFFFFFFu, mine.w, 1));
      uint8_t* const S = blk + (32 * (int64_t)kb + 8 * c + f) * n_e;
      const int a = (int)(reinterpret_cast<uintptr_t>(S) & 15u);
      if (own_end <= 0) continue;
      if (a == 0) {
        store_chunk(S + 16 * g, mine, 0, own_end);
      } else {
        const int o16 = 16 - a;
        // main chunk: tokens 16g + o16 .. 16g + o16 + 15
        const int valid = nv - (16 * g + o16);
        if (valid > 0) store_chunk(S + 16 * g + o16, window16(mine, next, o16), 0, valid);
        // head chunk (tokens 0 .. o16 - 1 at bytes a .. 15 of the chunk before S + o16)
        if (g == 0) store_chunk(S - a, window16(make_uint4(0u, 0u, 0u, 0u), mine, o16), a,
                                a + (nv < o16 ? nv : o16));
      }
    }
  }
}

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

fp4_status fp4_to_fp8_row(const uint8_t* packed, const uint8_t* scales, int64_t rows, int64_t cols,
                          uint8_t* fp8, float* fp8_scales, void* stream) {
  if (rows < 0 || cols < 0 || cols % 128 != 0) return FP4_ERR_SHAPE;
  const int64_t nspans = rows * (cols / 128);
  if (nspans > 0 && (!packed || !scales || !fp8 || !fp8_scales)) return FP4_ERR_NULL;
  if (!aligned(packed, 32) || !aligned(scales, 4) || !aligned(fp8, 32) || !aligned(fp8_scales, 4))
    return FP4_ERR_ALIGN;
  if (nspans == 0) return FP4_OK;
  return launch<fp4_to_fp8_row_kernel>(nspans, kRowThreads, 0, as_stream(stream), packed, scales,
                                       nspans, fp8, fp8_scales);
}

fp4_status fp4_to_fp8_col(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                          const int64_t* seg_row_off, const int64_t* seg_scale_off,
                          int32_t num_segments, int64_t total_rows, int64_t total_blocks,
                          uint8_t* fp8_t, float* fp8_t_scales, void* stream) {
  if (cols < 0 || cols % 128 != 0 || num_segments < 0 || total_rows < 0 || total_blocks < 0)
    return FP4_ERR_SHAPE;
  if (total_blocks > total_rows / 128 + num_segments) return FP4_ERR_SHAPE;
  if (!seg_row_off || !seg_scale_off) return FP4_ERR_NULL;
  const int64_t ntiles = total_blocks * (cols / 128);
  if (ntiles > 0 && (!packed || !scales || !fp8_t || !fp8_t_scales)) return FP4_ERR_NULL;
  if (!aligned(packed, 32) || !aligned(scales, 4) || !aligned(fp8_t_scales, 4) ||
      !aligned(seg_row_off, 8) || !aligned(seg_scale_off, 8))
    return FP4_ERR_ALIGN;
  if (ntiles == 0 || num_segments == 0) return FP4_OK;
  // one warp per (token block, 32-feature block), grid-stride over them
  const int64_t nunits = total_blocks * (cols / 32);
  return launch<fp4_to_fp8_col_kernel>(nunits * 32, kColThreads, 0, as_stream(stream), packed,
                                       scales, cols, seg_row_off, seg_scale_off, num_segments,
                                       nunits, fp8_t, fp8_t_scales);
}

}  // extern "C"
