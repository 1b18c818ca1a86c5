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
// transpose and requantize, with a padded shared-memory tile against bank
// conflicts, over ragged per-expert row segments located by precomputed
// offsets.
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

constexpr int kColThreads = 256;
constexpr int kInRowWords = 20;  // 64 B of codes + 16 B pad per token row

// Physical word of logical word `w` in output-tile row `row` (XOR swizzle
// that keeps both the transposed writes and the row reads conflict-free).
__device__ __forceinline__ int out_word(int row, int w) { return w ^ (((row >> 3) & 15) << 1); }

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

struct ColTile {
  int64_t row0;     // first source row of the segment
  int64_t n_e;      // tokens in the segment
  int64_t sofs;     // segment's first global token block
  int64_t b;        // token block within the segment
};

__global__ void __launch_bounds__(kColThreads)
    fp4_to_fp8_col_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                          int64_t cols, const int64_t* __restrict__ seg_row_off,
                          const int64_t* __restrict__ seg_scale_off, int nseg, int64_t ntiles,
                          uint8_t* __restrict__ fp8_t, float* __restrict__ fp8_t_scales) {
  __shared__ __align__(16) uint32_t in_tile[128 * kInRowWords];
  __shared__ __align__(16) uint32_t out_tile[128 * 32];
  __shared__ uint32_t sc_tile[128];
  __shared__ uint32_t warp_st[4];
  __shared__ __align__(8) uint8_t lut[128];
  __shared__ ColTile tile;

  build_shift_tables(lut);
  const uint2* lut2 = reinterpret_cast<const uint2*>(lut);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t ftiles = cols / 128;
  const int64_t row_bytes = cols / 2, row_scales = cols / 32;

  for (int64_t tid = blockIdx.x; tid < ntiles; tid += gridDim.x) {
    const int64_t fb = tid / ftiles;  // global token block
    const int64_t f = tid - fb * ftiles;  // feature tile (128 features)
    if (warp == 0) {
      const int e = find_segment(seg_scale_off, nseg, fb);
      if (lane == 0) {
        tile.row0 = seg_row_off[e];
        tile.n_e = seg_row_off[e + 1] - tile.row0;
        tile.sofs = seg_scale_off[e];
        tile.b = fb - tile.sofs;
      }
    }
    __syncthreads();  // tile (and, first time, lut) visible; previous tile's smem free
    const int64_t row0 = tile.row0, n_e = tile.n_e, b = tile.b;
    const int64_t nb_e = (n_e + 127) / 128;
    const int nv = (int)((n_e - 128 * b) < 128 ? (n_e - 128 * b) : 128);  // valid tokens
    const int64_t src_row = row0 + 128 * b;

    // Stage the 128 x 64 B code tile (two threads per token row) and the
    // 128 x 4 scale bytes; rows past the segment end read as zero.
    {
      const int r = t >> 1, h = t & 1;
      U32x8 v;
      if (r < nv) {
        v = ld_stream_v8(packed + (src_row + r) * row_bytes + 64 * f + 32 * h);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v.w[i] = 0u;
      }
      uint4* dst = reinterpret_cast<uint4*>(in_tile + r * kInRowWords + 8 * h);
      dst[0] = make_uint4(v.w[0], v.w[1], v.w[2], v.w[3]);
      dst[1] = make_uint4(v.w[4], v.w[5], v.w[6], v.w[7]);
      if (t < 128) {
        const uint32_t s = t < nv ? ld_stream_u32(scales + (src_row + t) * row_scales + 4 * f) : 0u;
        sc_tile[t] = s;
        // per-byte max over the block's tokens: S_t of the 4 feature blocks
        uint32_t m = s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = __vmaxu4(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) warp_st[warp] = m;
      }
    }
    __syncthreads();
    const uint32_t st4 = __vmaxu4(__vmaxu4(warp_st[0], warp_st[1]), __vmaxu4(warp_st[2], warp_st[3]));

    // Output scales: feature k of this tile, token block b.
    if (t < 128) {
      const uint32_t st = (st4 >> (8 * (t >> 5))) & 0xFFu;
      fp8_t_scales[cols * tile.sofs + (128 * f + t) * nb_e + b] = ue8m0_to_f32(st);
    }

    // Convert and transpose: lane owns word column c (features 8c..8c+7)
    // for token quads tq and tq + 16.
    {
      const int c = lane & 15;
      const int kb = c >> 2;
      const uint32_t st = (st4 >> (8 * kb)) & 0xFFu;
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int tq = 2 * warp + (lane >> 4) + 16 * rep;
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = 4 * tq + i;
          const uint32_t w = in_tile[j * kInRowWords + c];
          uint32_t d = st - ((sc_tile[j] >> (8 * kb)) & 0xFFu);
          d = d > 15u ? 15u : d;
          convert8(w, lut2[d], lo[i], hi[i]);
        }
        // 4x4 byte transposes: token-major words -> feature-major words
        const uint32_t a0 = __byte_perm(lo[0], lo[1], 0x5140u), a1 = __byte_perm(lo[0], lo[1], 0x7362u);
        const uint32_t a2 = __byte_perm(lo[2], lo[3], 0x5140u), a3 = __byte_perm(lo[2], lo[3], 0x7362u);
        const uint32_t b0 = __byte_perm(hi[0], hi[1], 0x5140u), b1 = __byte_perm(hi[0], hi[1], 0x7362u);
        const uint32_t b2 = __byte_perm(hi[2], hi[3], 0x5140u), b3 = __byte_perm(hi[2], hi[3], 0x7362u);
        uint32_t o[8];
        o[0] = __byte_perm(a0, a2, 0x5410u);
        o[1] = __byte_perm(a0, a2, 0x7632u);
        o[2] = __byte_perm(a1, a3, 0x5410u);
        o[3] = __byte_perm(a1, a3, 0x7632u);
        o[4] = __byte_perm(b0, b2, 0x5410u);
        o[5] = __byte_perm(b0, b2, 0x7632u);
        o[6] = __byte_perm(b1, b3, 0x5410u);
        o[7] = __byte_perm(b1, b3, 0x7632u);
#pragma unroll
        for (int fi = 0; fi < 8; ++fi) {
          const int row = 8 * c + fi;
          out_tile[row * 32 + out_word(row, tq)] = o[fi];
        }
      }
    }
    __syncthreads();

    // Store: each warp writes 16 feature rows; a row is nv bytes at an
    // arbitrary byte address, written as aligned 32-bit words (bytes at the
    // two ragged ends).
    for (int rr = 0; rr < 16; ++rr) {
      const int row = 16 * warp + rr;
      uint8_t* dst = fp8_t + cols * row0 + (128 * f + row) * n_e + 128 * b;
      const int a = (int)(reinterpret_cast<uintptr_t>(dst) & 3u);
      uint8_t* base = dst - a;
      const int nwords = (a + nv + 3) >> 2;
      for (int wi = lane; wi < nwords; wi += 32) {
        const int t0 = 4 * wi - a;  // tile byte held by the word's first byte
        uint32_t val;
        if (a == 0) {
          val = out_tile[row * 32 + out_word(row, wi)];
        } else {
          const uint32_t lo = wi >= 1 ? out_tile[row * 32 + out_word(row, wi - 1)] : 0u;
          const uint32_t hi = wi < 32 ? out_tile[row * 32 + out_word(row, wi)] : 0u;
          val = __funnelshift_r(lo, hi, 8 * (4 - a));
        }
        if (t0 >= 0 && t0 + 3 < nv) {
          *reinterpret_cast<uint32_t*>(base + 4 * wi) = val;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (t0 + q >= 0 && t0 + q < nv) base[4 * wi + q] = (uint8_t)(val >> (8 * q));
        }
      }
    }
    // the __syncthreads at the top of the next tile orders these reads
    // before the next tile's shared-memory writes
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
  // one CTA per tile, grid-stride over tiles
  static const int occ = occupancy(fp4_to_fp8_col_kernel, kColThreads, 0);
  int64_t grid = (int64_t)sm_count() * occ;
  if (grid > ntiles) grid = ntiles;
  fp4_to_fp8_col_kernel<<<(unsigned)grid, kColThreads, 0, as_stream(stream)>>>(
      packed, scales, cols, seg_row_off, seg_scale_off, num_segments, ntiles, fp8_t, fp8_t_scales);
  return after_launch();
}

}  // extern "C"
