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
// Work unit: one warp converts one 32-feature block (one MXFP4 scale column)
// over a run of up to kColRun consecutive 128-token blocks of the global
// block order (a run may cross segment boundaries).  Per token block:
//   - lane (g, c) = (lane >> 1, lane & 1) loads the 16 codes of features
//     16c .. 16c+15 (8 bytes) and the scale byte of tokens 8g .. 8g+7;
//   - the block's target scale S_t is one warp max reduction;
//   - each lane converts its 8 tokens x 16 features through the shift
//     tables and transposes them (4 x 4 byte transposes) into 16 feature
//     rows x 8 token bytes, written to the warp's tile in shared memory
//     (32 feature rows of 128 token bytes);
//   - the warp then writes the 32 rows, four at a time, eight lanes per row
//     each storing one aligned 16-byte chunk of the row's output span.  A
//     row's output start D is byte-aligned only, so each chunk is a window
//     of two aligned tile pieces, and the row's last (D mod 16) bytes are
//     carried, in a 16-byte slot before the row, to the next block of the
//     same segment.
// Inside a run every chunk is whole.  For a segment wholly inside the run,
// the warp's 32 output rows are one contiguous byte range, so the partial
// chunk where row r ends is the one where row r + 1 starts: the segment's
// first block keeps each row's head chunk and its last block stores it
// merged with the previous row's tail as one whole chunk; only the two ends
// of the range, shared with other warps, go out byte by byte.  Where a
// segment crosses a run's end (or has rows under 32 bytes), the partial
// chunks there are clipped and stored as words and bytes.
// No CTA barrier in the loop: the warps of a CTA are independent.  The 8
// warps of a CTA take neighbouring feature blocks of the same run, so their
// 16-byte row slices of the codes share one 128-byte line and their scale
// bytes one sector: those loads are cached in L1, so a line leaves L2 once
// per CTA rather than once per warp.

constexpr int kColThreads = 256;
constexpr int kColRun = 32;      // token blocks per unit
constexpr int kTileRow = 36;     // tile words per feature row: 4 carry words, 32 data words

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

// Bytes o .. o+15 (1 <= o <= 16) of the 32-byte sequence x[0..3] | y[0..3].
__device__ __forceinline__ uint4 window16(uint4 x, uint4 y, uint32_t o) {
  uint32_t w0 = x.x, w1 = x.y, w2 = x.z, w3 = x.w, w4 = y.x, w5 = y.y, w6 = y.z, w7 = y.w;
  if (o & 16u) return y;
  if (o & 8u) {
    w0 = w2; w1 = w3; w2 = w4; w3 = w5; w4 = w6; w5 = w7;
  }
  if (o & 4u) {
    w0 = w1; w1 = w2; w2 = w3; w3 = w4; w4 = w5;
  }
  const uint32_t sh = 8u * (o & 3u);
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                    __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// 4 x 4 byte transpose: x[i] holds bytes (i, 0..3); y[j] receives (0..3, j).
__device__ __forceinline__ void transpose4(const uint32_t x[4], uint32_t y[4]) {
  const uint32_t a0 = __byte_perm(x[0], x[1], 0x5140u), a1 = __byte_perm(x[0], x[1], 0x7362u);
  const uint32_t a2 = __byte_perm(x[2], x[3], 0x5140u), a3 = __byte_perm(x[2], x[3], 0x7362u);
  y[0] = __byte_perm(a0, a2, 0x5410u);
  y[1] = __byte_perm(a0, a2, 0x7632u);
  y[2] = __byte_perm(a1, a3, 0x5410u);
  y[3] = __byte_perm(a1, a3, 0x7632u);
}

// Bytes lo .. hi-1 (0 <= lo < hi <= 16) of the 16-byte value v to the
// 16-byte aligned p: one 128-bit store when the chunk is whole, otherwise
// the whole 32-bit words inside [lo, hi) as word stores and the bytes of
// the (at most two) edge words as byte stores.
__device__ __forceinline__ void store_chunk(uint8_t* p, uint4 v, int lo, int hi) {
  if (lo == 0 && hi == 16) {
    *reinterpret_cast<uint4*>(p) = v;
    return;
  }
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int b0 = 4 * t;
    if (lo <= b0 && b0 + 4 <= hi) {
      reinterpret_cast<uint32_t*>(p)[t] = vw[t];
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (b0 + q >= lo && b0 + q < hi) p[b0 + q] = (uint8_t)(vw[t] >> (8 * q));
    }
  }
}

// The segment holding a token block, walked forward block by block.
struct SegPos {
  int e;
  int64_t sofs, send;  // its blocks: [sofs, send)
  int64_t row0, n_e;   // its rows
};

__device__ __forceinline__ void seg_load(SegPos& p, const int64_t* __restrict__ row_off,
                                         const int64_t* __restrict__ scale_off) {
  p.sofs = scale_off[p.e];
  p.send = scale_off[p.e + 1];
  p.row0 = row_off[p.e];
  p.n_e = row_off[p.e + 1] - p.row0;
}

// Moves p forward to the segment holding block fb (warp-uniform); false if
// the offsets end before fb.
__device__ __forceinline__ bool seg_advance(SegPos& p, int64_t fb, int nseg,
                                            const int64_t* __restrict__ row_off,
                                            const int64_t* __restrict__ scale_off) {
  while (fb >= p.send && p.e + 1 < nseg) {
    ++p.e;
    seg_load(p, row_off, scale_off);
  }
  return fb < p.send;
}

// Codes (16 features) and scale bytes of a lane's 8 tokens of one block.
struct ColIn {
  uint2 w[8];
  uint32_t s[8];
};

__device__ __forceinline__ void col_issue(ColIn& in, const uint8_t* __restrict__ packed,
                                          const uint8_t* __restrict__ scales, const SegPos& p,
                                          int64_t fb, int64_t row_bytes, int64_t kblocks, int kb,
                                          int g, int c) {
  const int64_t t0 = 128 * (fb - p.sofs);
  const int64_t left = p.n_e - t0 - 8 * g;  // tokens of this lane's 8 that exist
  const int64_t r = p.row0 + t0 + 8 * g;
  const uint8_t* pw = packed + r * row_bytes + 16 * kb + 8 * c;
  const uint8_t* ps = scales + r * kblocks + kb;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool ok = i < left;
    in.w[i] = ok ? ld_shared_v2(pw + i * row_bytes) : make_uint2(0u, 0u);
    in.s[i] = ok ? ld_shared_u8(ps + i * kblocks) : 0u;
  }
}

// Converts and writes one token block of one 32-feature block (see above).
__device__ __forceinline__ void col_block(const ColIn& in, const SegPos& p, int64_t fb, bool carry,
                                          bool run_end, bool merge, int64_t cols, int kb, int lane,
                                          int g, int c, const uint2* lut2, uint32_t* tile,
                                          uint4* heads, uint8_t* __restrict__ fp8_t,
                                          float* __restrict__ fp8_t_scales) {
  const int64_t b = fb - p.sofs;  // block inside the segment
  const int64_t t0 = 128 * b;
  const int nv = p.n_e - t0 < 128 ? (int)(p.n_e - t0) : 128;  // tokens in this block
  uint32_t st = in.s[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) st = max(st, in.s[i]);
  st = __reduce_max_sync(0xFFFFFFFFu, st);
  fp8_t_scales[cols * p.sofs + (32 * kb + lane) * (p.send - p.sofs) + b] = ue8m0_to_f32(st);

  // Convert and transpose into the tile: row 16c + f, token bytes 8g .. 8g+7.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t x[4][4];  // x[i][k]: token 4h+i, features 4k .. 4k+3
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t d = st - in.s[4 * h + i];
      d = d > 15u ? 15u : d;
      const uint2 l = lut2[d];
      convert8(in.w[4 * h + i].x, l, x[i][0], x[i][1]);
      convert8(in.w[4 * h + i].y, l, x[i][2], x[i][3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t xi[4] = {x[0][k], x[1][k], x[2][k], x[3][k]};
      uint32_t y[4];
      transpose4(xi, y);
#pragma unroll
      for (int j = 0; j < 4; ++j) tile[(16 * c + 4 * k + j) * kTileRow + 4 + 2 * g + h] = y[j];
    }
  }
  __syncwarp();

  // Store the 32 rows: row r of this block covers output bytes
  // [D, D + nv), D = fp8_t + cols*row0 + (32kb + r)*n_e + t0.  A tile row
  // holds 16 carry bytes (bytes 112..127 of the previous block of the
  // segment) and then the block's 128 bytes.
  uint8_t* const D0 = fp8_t + cols * p.row0 + 32 * kb * p.n_e + t0;
  if (carry && !run_end) {
    // every chunk whole: row r writes the aligned 16-byte chunks j = 0..7
    // of [D - a, D - a + 128), a = D mod 16, lanes 8q + j of step i take
    // row 4i + q
    const int q = lane >> 3, j = lane & 7;
#pragma unroll 4
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + q;
      uint8_t* const D = D0 + (int64_t)r * p.n_e;
      const uint32_t a = (uint32_t)reinterpret_cast<uintptr_t>(D) & 15u;
      const uint4* row = reinterpret_cast<const uint4*>(tile + r * kTileRow);  // row[0]: carry
      reinterpret_cast<uint4*>(D - a)[j] = window16(row[j], row[j + 1], 16u - a);
    }
  } else if (merge) {
    // first or last block of a segment whose rows are at least 32 bytes:
    // the row's span in chunk coordinates u = x + a is [ulo, uhi); its
    // whole chunks go out as above.  A row's partial head chunk (first
    // block) is kept in heads[r]: the same 16 bytes hold the end of row
    // r - 1, and the last block stores the two merged as one whole chunk.
    // Only row 0's head and row 31's tail border other warps' rows; those
    // bytes go out one at a time.
    const int q = lane >> 3, j = lane & 7;
#pragma unroll 4
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + q;
      uint8_t* const D = D0 + (int64_t)r * p.n_e;
      const uint32_t a = (uint32_t)reinterpret_cast<uintptr_t>(D) & 15u;
      const int ulo = carry ? 0 : (int)a;
      const int uhi = run_end ? nv + (int)a : 128;
      if (16 * j >= ulo && 16 * j + 16 <= uhi) {
        const uint4* row = reinterpret_cast<const uint4*>(tile + r * kTileRow);  // row[0]: carry
        reinterpret_cast<uint4*>(D - a)[j] = window16(row[j], row[j + 1], 16u - a);
      }
    }
    uint8_t* const D = D0 + (int64_t)lane * p.n_e;
    const uint32_t a = (uint32_t)reinterpret_cast<uintptr_t>(D) & 15u;
    uint8_t* const G = D - a;  // byte u of the span is G[u]
    const uint4* row = reinterpret_cast<const uint4*>(tile + lane * kTileRow);
    if (!carry && a != 0u) {  // head chunk 0: bytes [a, 16) are this row's
      const uint4 h = window16(row[0], row[1], 16u - a);
      if (lane == 0) {
        const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
        for (int m = 0; m < 16; ++m)
          if (m >= (int)a) G[m] = (uint8_t)(hw[m >> 2] >> (8 * (m & 3)));
      } else {
        heads[lane] = h;
      }
    }
    __syncwarp();
    if (run_end) {
      const int uhi = nv + (int)a;
      const int kt = uhi >> 4, tl = uhi & 15;  // tail chunk kt: bytes [0, tl) are this row's
      if (tl != 0) {
        const uint4 nxt = kt < 8 ? row[kt + 1] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 t = window16(row[kt], nxt, 16u - a);
        if (lane < 31) {
          // the rest of the chunk is the head of row r + 1 (it starts at
          // byte tl of this chunk): one whole chunk
          const uint4 h = heads[lane + 1];
          const uint32_t tw[4] = {t.x, t.y, t.z, t.w}, hw[4] = {h.x, h.y, h.z, h.w};
          uint32_t mw[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int lo = tl - 4 * w;  // bytes of word w taken from the tail
            const uint32_t keep = lo >= 4 ? 0xFFFFFFFFu : (lo <= 0 ? 0u : (1u << (8 * lo)) - 1u);
            mw[w] = (tw[w] & keep) | (hw[w] & ~keep);
          }
          reinterpret_cast<uint4*>(G)[kt] = make_uint4(mw[0], mw[1], mw[2], mw[3]);
        } else {
          const uint32_t tw[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
          for (int m = 0; m < 16; ++m)
            if (m < tl) G[16 * kt + m] = (uint8_t)(tw[m >> 2] >> (8 * (m & 3)));
        }
      }
    }
  } else {
    // first or last block of a segment with rows shorter than 32 bytes: the
    // same chunks (nine when the span ends past chunk 7), each clipped to
    // the row bytes [lo, hi) this block writes
    const int q = lane >> 3, j = lane & 7;
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + q;
      uint8_t* const D = D0 + (int64_t)r * p.n_e;
      const int a = (int)(reinterpret_cast<uintptr_t>(D) & 15u);
      const int lo = carry ? -a : 0;  // without carry the bytes before t0 are not ours
      const int hi = run_end ? nv : 128 - a;
      const uint4* row = reinterpret_cast<const uint4*>(tile + r * kTileRow);
#pragma unroll
      for (int k = j; k < 9; k += 8) {  // chunk k: row bytes [16k - a, 16k - a + 16)
        const int c0 = 16 * k - a;
        const int blo = lo - c0 > 0 ? lo - c0 : 0;
        const int bhi = hi - c0 < 16 ? hi - c0 : 16;
        if (blo < bhi) {
          const uint4 nxt = k + 1 < 9 ? row[k + 1] : make_uint4(0u, 0u, 0u, 0u);
          store_chunk(D - a + 16 * k, window16(row[k], nxt, 16u - (uint32_t)a), blo, bhi);
        }
      }
    }
  }
  __syncwarp();
  if (!run_end) {  // carry: lane r copies row r's last 16 bytes
    uint4* row = reinterpret_cast<uint4*>(tile + lane * kTileRow);
    row[0] = row[8];
  }
  __syncwarp();
}

// The loads of the next token block are issued before the current one is
// converted and written (two register buffers, swapped by unrolling).  A
// segment that lies wholly inside the run (and has rows of 32 bytes or
// more) merges its row ends; one that crosses the run's ends writes the
// partial chunks there byte by byte.
__global__ void __launch_bounds__(kColThreads)
    fp4_to_fp8_col_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                          int64_t cols, const int64_t* __restrict__ seg_row_off,
                          const int64_t* __restrict__ seg_scale_off, int nseg, int64_t total_blocks,
                          int64_t nunits, uint8_t* __restrict__ fp8_t,
                          float* __restrict__ fp8_t_scales) {
  __shared__ __align__(8) uint8_t lut[128];
  __shared__ __align__(16) uint32_t tiles[kColThreads / 32][32 * kTileRow];
  __shared__ uint4 head_tiles[kColThreads / 32][32];
  build_shift_tables(lut);
  __syncthreads();
  const uint2* lut2 = reinterpret_cast<const uint2*>(lut);
  uint32_t* const tile = tiles[threadIdx.x >> 5];
  uint4* const heads = head_tiles[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const int g = lane >> 1;  // tokens 8g .. 8g+7 of a block
  const int c = lane & 1;   // features 16c .. 16c+15 of the feature block
  const int64_t kblocks = cols / 32;
  const int64_t row_bytes = cols / 2;
  const int64_t nwarps = (int64_t)gridDim.x * (kColThreads / 32);
  for (int64_t unit = (int64_t)blockIdx.x * (kColThreads / 32) + (threadIdx.x >> 5); unit < nunits;
       unit += nwarps) {
    const int64_t run = unit / kblocks;
    const int kb = (int)(unit - run * kblocks);
    const int64_t fb0 = run * kColRun;
    const int64_t fb1 = fb0 + kColRun < total_blocks ? fb0 + kColRun : total_blocks;
    SegPos pa;
    pa.e = find_segment(seg_scale_off, nseg, fb0);
    seg_load(pa, seg_row_off, seg_scale_off);
    if (!seg_advance(pa, fb0, nseg, seg_row_off, seg_scale_off)) continue;
    ColIn A, B;
    col_issue(A, packed, scales, pa, fb0, row_bytes, kblocks, kb, g, c);
    SegPos pb = pa;
    for (int64_t fb = fb0;;) {
      // A holds block fb (segment pa); fetch fb + 1 into B
      bool next = fb + 1 < fb1;
      pb = pa;
      if (next) next = seg_advance(pb, fb + 1, nseg, seg_row_off, seg_scale_off);
      if (next) col_issue(B, packed, scales, pb, fb + 1, row_bytes, kblocks, kb, g, c);
      col_block(A, pa, fb, fb != fb0 && fb != pa.sofs, !next || fb + 1 == pa.send,
                pa.sofs >= fb0 && pa.send <= fb1 && pa.n_e >= 32, cols, kb, lane, g, c, lut2, tile,
                heads, fp8_t, fp8_t_scales);
      if (!next) break;
      ++fb;
      // B holds block fb (segment pb); fetch fb + 1 into A
      next = fb + 1 < fb1;
      pa = pb;
      if (next) next = seg_advance(pa, fb + 1, nseg, seg_row_off, seg_scale_off);
      if (next) col_issue(A, packed, scales, pa, fb + 1, row_bytes, kblocks, kb, g, c);
      col_block(B, pb, fb, fb != fb0 && fb != pb.sofs, !next || fb + 1 == pb.send,
                pb.sofs >= fb0 && pb.send <= fb1 && pb.n_e >= 32, cols, kb, lane, g, c, lut2, tile,
                heads, fp8_t, fp8_t_scales);
      if (!next) break;
      ++fb;
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
  // one warp per (run of kColRun token blocks, 32-feature block)
  const int64_t nunits = (total_blocks + kColRun - 1) / kColRun * (cols / 32);
  return launch<fp4_to_fp8_col_kernel>(nunits * 32, kColThreads, 0, as_stream(stream), packed,
                                       scales, cols, seg_row_off, seg_scale_off, num_segments,
                                       total_blocks, nunits, fp8_t, fp8_t_scales);
}

}  // extern "C"
