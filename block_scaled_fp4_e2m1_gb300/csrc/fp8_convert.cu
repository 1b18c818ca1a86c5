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
// Output: for expert segment e (rows row0 .. row0 + n_e - 1 of the input),
// feature f's n_e E4M3 bytes at fp8_t + cols * row0 + f * n_e.  Rows start
// at arbitrary byte offsets, so the stores are organised around 32-byte
// sectors: every store covers whole sectors, and a sector shared by two
// rows is written once, merged.  (Measured: the same 16-byte stores ran
// 14% faster when moved to 32-byte alignment, where they no longer left
// sectors half written.)
//
// Work unit: one CTA converts a group of up to eight 32-feature blocks (one
// MXFP4 scale column each, one per warp) over a run of consecutive 128-token
// blocks of the global block order (a run may cross segment boundaries).
// The run length is chosen per launch (col_run_blocks) so that the units
// fill whole waves of resident CTAs.  Per token block:
//   - the CTA copies the block's codes for its 256 features (128 tokens x
//     128 bytes: whole lines) and their scale bytes into a shared-memory
//     stage with cp.async, one block ahead of use; 16-byte chunk q of token
//     t sits at chunk q ^ ((t >> 3) & 7) of its row, so the warps' reads
//     are free of bank conflicts;
//   - in warp w (feature block w of the group) lane (g, c) = (lane >> 1,
//     lane & 1) reads the 16 codes of features 16c .. 16c+15 and the scale
//     byte of tokens 8g .. 8g+7 from the stage;
//   - the block's target scale S_t is one warp max reduction;
//   - each lane converts its 8 tokens x 16 features through the shift
//     tables and transposes them (4 x 4 byte transposes) into 16 feature
//     rows x 8 token bytes of the warp's tile in shared memory: 32 rows of
//     a 32-byte carry (the previous block's last 32 tokens) and the block's
//     128 token bytes (rows 16 .. 31 start 64 bytes further on, so the two
//     halves of the warp write different banks);
//   - four lanes per row store the row's whole sectors that this block
//     completes, each a 32-byte window of the tile row; the row's last
//     (partial) sector is left to the next block through the carry.
// At a segment's first block a row's first, partial sector (it begins
// with the end of the previous row) is skipped, and the row's first 32
// bytes are kept as its head.  At the segment's last block, lane r stores
// row r's last partial sector merged with the head of row r + 1 (the next
// warp's row 0 for r = 31).  Only where a CTA's group of features begins
// and ends do partial sectors go out byte by byte.
// A unit that starts inside a segment first converts, without storing,
// the block before its run (for the carry) and, if the segment ends within
// the run, the segment's first block (for the heads).  A segment under 32
// tokens is one contiguous span of the CTA's rows: they are laid out in
// order in shared memory and the span goes out as whole sectors
// (col_store_short).
// One CTA barrier per token block publishes a stage and frees the one read
// before; a segment of one block adds one between its heads and merges.
// Token-block indices are 32-bit (the host admits fewer than 2^31 blocks);
// row offsets stay 64-bit.

constexpr int kColThreads = 256;
constexpr int kColGroup = kColThreads / 32;  // feature blocks per CTA: one per warp
constexpr int kColRunMin = 8;   // token blocks per unit: at least
constexpr int kColRunMax = 40;  // and at most (a unit converts up to two
                                // extra blocks for its carry and heads)
constexpr int kColRunLimit = 1 << 20;  // largest run a caller may fix
constexpr int kStageCodes = 128 * 16 * kColGroup;  // code bytes of one stage
constexpr int kStageBytes = kStageCodes + 128 * kColGroup;  // + scale bytes
// tile words per feature row: 8 carry words, 32 data words, 4 words of
// padding (a pitch of 44 words puts 8 consecutive rows' 16-byte chunks in
// different banks)
constexpr int kTileRow = 44;
constexpr int kTileWords = 32 * kTileRow + 16;  // rows 16 .. 31 shifted by 16 words
constexpr int kHeadWords = 32 * 8;              // heads: 32 rows x 32 bytes
// Segment offsets held in shared memory (entries of each table): with up
// to kSegTab - 1 segments the CTA copies both offset tables once, so the
// segment walk and the search at each unit's start read shared memory
// instead of waiting on global loads (2-7% faster on the MoE workloads).
constexpr int kSegTab = 512;
constexpr size_t kColSmem = 2 * (size_t)kStageBytes +
                            kColGroup * (kTileWords + kHeadWords) * 4 + 2 * 8 * kSegTab + 128;

// Row r of a warp's tile, as 10 16-byte chunks: 0-1 carry, 2-9 data.
__device__ __forceinline__ uint4* tile_row(uint32_t* tile, int r) {
  return reinterpret_cast<uint4*>(tile + r * kTileRow + (r >= 16 ? 16 : 0));
}

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

// Bytes o .. o+15 (0 <= o <= 16) of the 32-byte sequence x[0..3] | y[0..3].
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

// Bytes o .. o+31 (0 <= o <= 32) of the 64-byte sequence w[0..15], into
// r[0..7].
__device__ __forceinline__ void window32(const uint32_t w[16], uint32_t o, uint32_t r[8]) {
  if (o & 32u) {  // the second half, whole
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = w[8 + k];
    return;
  }
  // v[0..8] = w[(o >> 2) .. (o >> 2) + 8], by shifts of 4, 2 and 1 words
  uint32_t v[12];
#pragma unroll
  for (int k = 0; k < 12; ++k) v[k] = (o & 16u) ? w[k + 4] : w[k];
#pragma unroll
  for (int k = 0; k < 10; ++k) v[k] = (o & 8u) ? v[k + 2] : v[k];
#pragma unroll
  for (int k = 0; k < 9; ++k) v[k] = (o & 4u) ? v[k + 1] : v[k];
  const uint32_t sh = 8u * (o & 3u);
#pragma unroll
  for (int k = 0; k < 8; ++k) r[k] = __funnelshift_r(v[k], v[k + 1], sh);
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

// Bytes [t_lo, t_hi) of tile row `row` (byte x holds token t0 - 32 + x) to
// dst[t - t_lo] one byte at a time.
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint4* row, int x_lo, int x_hi) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(row);
  for (int x = x_lo; x < x_hi; ++x) dst[x - x_lo] = (uint8_t)(w[x >> 2] >> (8 * (x & 3)));
}

// The segment holding a token block, walked forward block by block.
struct SegPos {
  int e;
  int sofs, send;      // its blocks: [sofs, send) (block indices < 2^31)
  int64_t row0, n_e;   // its rows
};

__device__ __forceinline__ void seg_load(SegPos& p, const int64_t* __restrict__ row_off,
                                         const int64_t* __restrict__ scale_off) {
  p.sofs = (int)scale_off[p.e];
  p.send = (int)scale_off[p.e + 1];
  p.row0 = row_off[p.e];
  p.n_e = row_off[p.e + 1] - p.row0;
}

// Moves p forward to the segment holding block fb (warp-uniform); false if
// the offsets end before fb.
__device__ __forceinline__ bool seg_advance(SegPos& p, int fb, int nseg,
                                            const int64_t* __restrict__ row_off,
                                            const int64_t* __restrict__ scale_off) {
  while (fb >= p.send && p.e + 1 < nseg) {
    ++p.e;
    seg_load(p, row_off, scale_off);
  }
  return fb < p.send;
}

// cp.async of `n` (16 or 4) bytes, the first `valid` of them from global
// memory and the rest zero (valid = 0: nothing is read).
template <int n>
__device__ __forceinline__ void cp_async_zfill(void* smem, const void* gmem, int valid) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  if (n == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(valid)
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(gmem), "r"(valid)
                 : "memory");
}

// The whole CTA copies token block fb of segment p for feature blocks
// 8grp .. 8grp + nkb - 1 into stage `stg`: codes (16-byte chunk q of token
// t at chunk q ^ ((t >> 3) & 7) of row t), then scale bytes (token t's from
// 8 * (16 * (t & 7) + (t >> 3)) on, so that the 16 tokens 8g + i, g = 0..15,
// a warp reads at once sit in different banks).  Missing tokens and feature
// blocks are zero.
__device__ __forceinline__ void col_stage(uint8_t* stg, const uint8_t* __restrict__ packed,
                                          const uint8_t* __restrict__ scales, const SegPos& p,
                                          int fb, int64_t row_bytes, int64_t kblocks, int grp,
                                          int nkb) {
  const int64_t t0 = 128 * (int64_t)(fb - p.sofs);
  const int nv = p.n_e - t0 < 128 ? (int)(p.n_e - t0) : 128;
  const int64_t r0 = p.row0 + t0;
  // copy k moves token tb + 32 k, chunk q: one base address plus k steps
  const int tb = (int)threadIdx.x >> 3, q = (int)threadIdx.x & 7;
  const uint8_t* src0 = packed + (r0 + tb) * row_bytes + 16 * (kColGroup * grp + q);
  const int64_t src_step = 32 * row_bytes;
  uint8_t* const dst0 = stg + 128 * tb + 16 * (q ^ (tb >> 3));
  uint8_t* const dst1 = stg + 128 * tb + 16 * (q ^ (tb >> 3) ^ 4);
  const bool qok = q < nkb;
#pragma unroll
  for (int k = 0; k < 128 * kColGroup / kColThreads; ++k) {
    const bool ok = tb + 32 * k < nv && qok;
    cp_async_zfill<16>((k & 1 ? dst1 : dst0) + 4096 * k, ok ? src0 + k * src_step : packed,
                       ok ? 16 : 0);
  }
  {
    // thread (i, g, h) = (tid >> 5, (tid >> 1) & 15, tid & 1): token 8g + i,
    // feature blocks 4h .. 4h+3
    const int i = (int)threadIdx.x >> 5, gg = ((int)threadIdx.x >> 1) & 15;
    const int h = (int)threadIdx.x & 1;
    const int t = 8 * gg + i;
    const bool ok = t < nv && 4 * h < nkb;
    const uint8_t* src = ok ? scales + (r0 + t) * kblocks + kColGroup * grp + 4 * h : scales;
    cp_async_zfill<4>(stg + kStageCodes + 8 * (16 * i + gg) + 4 * h, src, ok ? 4 : 0);
  }
}

// Converts staged token block b of a segment into the warp's tile (feature
// block kbl of the stage); returns S_t.  At the segment's first block it
// also keeps each row's first 32 bytes in heads.
__device__ __forceinline__ uint32_t col_convert(const uint8_t* stg, int kbl, int g, int c, int lane,
                                                bool keep_heads, const uint2* lut2,
                                                uint32_t* tile, uint4* heads) {
  uint2 w[8];
  uint32_t sc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = 8 * g + i;
    w[i] = *reinterpret_cast<const uint2*>(stg + 128 * t + 16 * (kbl ^ (g & 7)) + 8 * c);
    sc[i] = stg[kStageCodes + 8 * (16 * i + g) + kbl];
  }
  uint32_t st = sc[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) st = max(st, sc[i]);
  st = __reduce_max_sync(0xFFFFFFFFu, st);

  // Convert and transpose: row 16c + f gets token bytes 8g .. 8g+7 at data
  // words 2g (tokens 8g .. 8g+3) and 2g + 1.
  uint32_t y[2][4][4];  // y[h][k][j]: row 16c + 4k + j, tokens 8g+4h .. 8g+4h+3
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t x[4][4];  // x[i][k]: token 4h+i, features 4k .. 4k+3
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t d = st - sc[4 * h + i];
      d = d > 15u ? 15u : d;
      const uint2 l = lut2[d];
      convert8(w[4 * h + i].x, l, x[i][0], x[i][1]);
      convert8(w[4 * h + i].y, l, x[i][2], x[i][3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t xi[4] = {x[0][k], x[1][k], x[2][k], x[3][k]};
      transpose4(xi, y[h][k]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      reinterpret_cast<uint2*>(tile_row(tile, 16 * c + 4 * k + j))[4 + g] =
          make_uint2(y[0][k][j], y[1][k][j]);
  __syncwarp();
  if (keep_heads) {
    const uint4* row = tile_row(tile, lane);
    heads[2 * lane] = row[2];
    heads[2 * lane + 1] = row[3];
  }
  return st;
}

// Stores token block b of segment p from the warp's tile (rows
// R_r = base + r * n_e, block bytes from R_r + t0).  first / last: b is the
// segment's first / last block; own_head: this warp writes row 0's first
// partial sector (it begins a CTA's feature group); next_head: the head of
// the row after row 31 (null where that row is another CTA's: row 31's
// last partial sector is then written byte by byte).
__device__ __forceinline__ void col_store(uint32_t* tile, const uint4* heads,
                                          const uint4* next_head, uint8_t* base, int64_t n_e,
                                          int64_t t0, int nv, bool first, bool last, bool own_head,
                                          int lane) {
  // whole sectors: lane (q, s) = (lane >> 2, lane & 3) takes sector s of
  // [L', L' + 128) of row 8i + q, L' = A rounded down to a sector,
  // A = R_r + t0, as one 32-byte store
  const int q = lane >> 2, s = lane & 3;
#pragma unroll 2
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + q;
    uint8_t* const A = base + (int64_t)r * n_e + t0;
    const uint32_t a = (uint32_t)reinterpret_cast<uintptr_t>(A) & 31u;
    // sectors [lo, hi) of the window are this block's to write
    const int lo = first && a != 0u ? 1 : 0;
    const int hi = last ? (int)((a + (uint32_t)nv) >> 5) : 4;
    if (s >= lo && s < hi) {
      // the sector's first byte is tile byte off (1 <= off <= 128): words
      // off/4 .. off/4 + 8 of the row (the ninth, read only when off < 128
      // needs it, is at most word 40, the row's first padding word),
      // shifted down by off mod 4 bytes
      const uint32_t off = 32u - a + 32u * (uint32_t)s;
      const uint32_t* w = reinterpret_cast<const uint32_t*>(tile_row(tile, r)) + (off >> 2);
      uint32_t v[9];
#pragma unroll
      for (int j = 0; j < 9; ++j) v[j] = w[j];
      const uint32_t sh = 8u * (off & 3u);
      U32x8 o;
#pragma unroll
      for (int j = 0; j < 8; ++j) o.w[j] = __funnelshift_r(v[j], v[j + 1], sh);
      st_v8(A - a + 32 * s, o);
    }
  }
  const uint4* row = tile_row(tile, lane);
  if (first && own_head && lane == 0) {
    // row 0's first partial sector: bytes [A, A rounded up to a sector)
    const uint32_t a = (uint32_t)reinterpret_cast<uintptr_t>(base) & 31u;
    if (a != 0u) store_bytes(base, row, 32, 32 + (int)(32u - a));
  }
  if (last) {
    // row r's last partial sector [E - m, E), E = R_{r+1}, merged with the
    // first 32 - m bytes of row r + 1
    uint8_t* const E = base + (int64_t)(lane + 1) * n_e;
    const uint32_t m = (uint32_t)reinterpret_cast<uintptr_t>(E) & 31u;
    if (m != 0u) {
      const uint4* h = lane < 31 ? heads + 2 * (lane + 1) : next_head;
      if (h == nullptr) {
        store_bytes(E - m, row, 32 + nv - (int)m, 32 + nv);
      } else {
        // W = tile bytes [nv, nv + 32): the row's last 32 tokens
        const uint32_t k = (uint32_t)nv >> 4;
        const uint4 c0 = row[k], c1 = row[k + 1], c2 = row[k + 2 < 10 ? k + 2 : 9];
        const uint4 w0 = window16(c0, c1, (uint32_t)nv & 15u);
        const uint4 w1 = window16(c1, c2, (uint32_t)nv & 15u);
        const uint4 h0 = h[0], h1 = h[1];
        const uint32_t seq[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                                  h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        uint32_t rr[8];
        window32(seq, 32u - m, rr);
        uint4* const S = reinterpret_cast<uint4*>(E - m);
        S[0] = make_uint4(rr[0], rr[1], rr[2], rr[3]);
        S[1] = make_uint4(rr[4], rr[5], rr[6], rr[7]);
      }
    }
  }
}

// Stores a segment of n_e < 32 tokens (one block) for the CTA's nkb
// feature blocks.  Their rows are one contiguous span of 32 nkb n_e bytes
// from base (row r of warp w at base + (32 w + r) n_e), too short for
// whole sectors per row, so the rows are first laid out in order in lin
// (shared memory, the span's byte k at lin[p0 + k], p0 = base mod 32:
// global and shared addresses then agree mod 32), then the span goes out
// as whole 32-byte sectors, one per thread, and its partial first and last
// sectors (shared with the neighbouring spans) byte by byte.  The whole
// CTA calls it.
__device__ __forceinline__ void col_store_short(uint8_t* lin, const uint32_t* tile, uint8_t* base,
                                                int n_e, int nkb, int wid, int lane) {
  const uint32_t p0 = (uint32_t)reinterpret_cast<uintptr_t>(base) & 31u;
  if (wid < nkb) {
    // the row's n_e tokens are tile bytes 32 .. 32 + n_e - 1
    const uint4* row = tile_row(const_cast<uint32_t*>(tile), lane);
    const uint4 h0 = row[2], h1 = row[3];
    const uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint8_t* const dst = lin + p0 + (32 * wid + lane) * n_e;
#pragma unroll
    for (int x = 0; x < 31; ++x)
      if (x < n_e) dst[x] = (uint8_t)(w[x >> 2] >> (8 * (x & 3)));
  }
  __syncthreads();
  const int len = 32 * nkb * n_e;
  const int t = (int)threadIdx.x;
  const int head = (int)((32u - p0) & 31u) < len ? (int)((32u - p0) & 31u) : len;
  const int tail0 = (int)((p0 + (uint32_t)len) & ~31u) - (int)p0;  // last sector start, span byte
  const int tail = tail0 > head ? tail0 : head;
  if (t < (tail - head) >> 5) {  // sector t: span bytes head + 32 t ..
    const uint4* src = reinterpret_cast<const uint4*>(lin + p0 + head + 32 * t);
    const uint4 a = src[0], b = src[1];
    U32x8 o;
    o.w[0] = a.x; o.w[1] = a.y; o.w[2] = a.z; o.w[3] = a.w;
    o.w[4] = b.x; o.w[5] = b.y; o.w[6] = b.z; o.w[7] = b.w;
    st_v8(base + head + 32 * t, o);
  }
  if (t < head) base[t] = lin[p0 + t];
  if (t < len - tail) base[tail + t] = lin[p0 + tail + t];
}

// Block converted by item `it` of a unit (see the kernel).
__device__ __forceinline__ int col_item_block(int it, int npre, bool pre_head,
                                              const SegPos& p0, int fb0) {
  if (it < npre) return (pre_head && it == 0) ? p0.sofs : fb0 - 1;
  return fb0 + (it - npre);
}

// Stages item `it` into stage it & 1 (nothing past the run or the offsets)
// and commits its cp.async group; ps follows the staged blocks' segments.
__device__ __forceinline__ void col_stage_item(
    int it, int npre, bool pre_head, const SegPos& p0, SegPos& ps, int fb0, int fb1,
    uint8_t* stages, const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
    int64_t row_bytes, int64_t kblocks, int grp, int nkb, int nseg,
    const int64_t* __restrict__ row_off, const int64_t* __restrict__ scale_off) {
  const int fb = col_item_block(it, npre, pre_head, p0, fb0);
  bool ok = fb < fb1;
  if (ok && it >= npre) ok = seg_advance(ps, fb, nseg, row_off, scale_off);
  if (ok)
    col_stage(stages + (it & 1) * kStageBytes, packed, scales, it < npre ? SegPos(p0) : SegPos(ps),
              fb, row_bytes, kblocks, grp, nkb);
  cp_async_commit();
}

// A unit's token blocks, in order: up to two blocks that are only
// converted (the first segment's block 0 for the heads, the block before
// the run for the carry), then the run's blocks.  The CTA stages each block
// one ahead (one cp.async group per block, committed even when empty).
// kTab: the segment offsets are read from a copy in shared memory.
template <bool kTab>
__global__ void __launch_bounds__(kColThreads)
    fp4_to_fp8_col_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                          int64_t cols, const int64_t* __restrict__ g_row_off,
                          const int64_t* __restrict__ g_scale_off, int nseg, int64_t total_blocks,
                          int64_t run_len, int64_t nunits, uint8_t* __restrict__ fp8_t,
                          float* __restrict__ fp8_t_scales) {
  extern __shared__ __align__(16) uint8_t col_smem[];
  uint8_t* const stages = col_smem;
  uint32_t* const tiles = reinterpret_cast<uint32_t*>(col_smem + 2 * kStageBytes);
  uint4* const all_heads = reinterpret_cast<uint4*>(tiles + kColGroup * kTileWords);
  uint8_t* const lut = col_smem + kColSmem - 128;
  build_shift_tables(lut);
  int64_t* const tab = reinterpret_cast<int64_t*>(col_smem + kColSmem - 128 - 2 * 8 * kSegTab);
  const int64_t* seg_row_off = g_row_off;
  const int64_t* seg_scale_off = g_scale_off;
  if (kTab) {  // read after the unit loop's first barrier
    for (int i = threadIdx.x; i <= nseg; i += kColThreads) {
      tab[i] = g_row_off[i];
      tab[kSegTab + i] = g_scale_off[i];
    }
    seg_row_off = tab;
    seg_scale_off = tab + kSegTab;
  }
  const uint2* lut2 = reinterpret_cast<const uint2*>(lut);
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  uint32_t* const tile = tiles + wid * kTileWords;
  uint4* const heads = all_heads + wid * (kHeadWords / 4);
  const int g = lane >> 1;  // tokens 8g .. 8g+7 of a block
  const int c = lane & 1;   // features 16c .. 16c+15 of the feature block
  const int64_t kblocks = cols / 32;
  const int64_t row_bytes = cols / 2;
  const int64_t ngroups = (kblocks + kColGroup - 1) / kColGroup;
  for (int64_t unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
    __syncthreads();  // the previous unit is done with the stages and heads; tables built
    const int64_t run = unit / ngroups;
    const int grp = (int)(unit - run * ngroups);
    const int nkb = (int)(kblocks - kColGroup * grp < kColGroup ? kblocks - kColGroup * grp
                                                                : kColGroup);
    const int kb = kColGroup * grp + wid;
    const bool active = wid < nkb;
    const int fb0 = (int)(run * run_len);
    const int fb1 = (int)(run * run_len + run_len < total_blocks ? run * run_len + run_len
                                                                 : total_blocks);
    SegPos p0;
    p0.e = find_segment(seg_scale_off, nseg, fb0);
    seg_load(p0, seg_row_off, seg_scale_off);
    if (!seg_advance(p0, fb0, nseg, seg_row_off, seg_scale_off)) continue;
    const int blo = fb0 - p0.sofs;  // the run's first block inside its first segment
    const bool pre_head = blo > 1 && p0.send <= fb1 && p0.n_e >= 32;
    const int npre = (pre_head ? 1 : 0) + (blo > 0 ? 1 : 0);
    // item it converts block item_block(it) (items < npre are in segment p0)
    SegPos ps = p0;  // segment of the next block to stage
    col_stage_item(0, npre, pre_head, p0, ps, fb0, fb1, stages, packed, scales, row_bytes, kblocks,
                   grp, nkb, nseg, seg_row_off, seg_scale_off);
    SegPos p = p0;
    for (int it = 0;; ++it) {
      cp_async_wait<0>();
      __syncthreads();  // block it is staged; block it - 1 is read
      col_stage_item(it + 1, npre, pre_head, p0, ps, fb0, fb1, stages, packed, scales, row_bytes,
                     kblocks, grp, nkb, nseg, seg_row_off, seg_scale_off);
      const bool real = it >= npre;
      const int fb = col_item_block(it, npre, pre_head, p0, fb0);
      if (real && !seg_advance(p, fb, nseg, seg_row_off, seg_scale_off)) break;
      const SegPos sp = real ? p : p0;
      const int b = fb - sp.sofs;
      const int64_t t0 = 128 * (int64_t)b;
      const int nv = sp.n_e - t0 < 128 ? (int)(sp.n_e - t0) : 128;
      const bool first = b == 0, last = fb + 1 == sp.send;
      const uint8_t* const stg = stages + (it & 1) * kStageBytes;
      if (active) {
        const uint32_t st = col_convert(stg, wid, g, c, lane, first && sp.n_e >= 32, lut2, tile,
                                        heads);
        if (real)
          fp8_t_scales[cols * sp.sofs + (int64_t)(32 * kb + lane) * (sp.send - sp.sofs) + b] =
              ue8m0_to_f32(st);
      }
      if (real && sp.n_e < 32) {
        // a short segment: the CTA's rows through the heads area, in order
        col_store_short(reinterpret_cast<uint8_t*>(all_heads),
                        tile,
                        fp8_t + cols * sp.row0 + 32 * kColGroup * grp * sp.n_e, (int)sp.n_e, nkb,
                        wid, lane);
      } else {
        // heads kept at this very block must be visible to the warp before
        // (heads of an earlier block are, through the barrier above)
        if (real && last && first) __syncthreads();
        if (active && real) {
          uint8_t* const base = fp8_t + cols * sp.row0 + 32 * kb * sp.n_e;
          const uint4* next_head =
              wid + 1 < nkb ? all_heads + (wid + 1) * (kHeadWords / 4) : nullptr;
          col_store(tile, heads, next_head, base, sp.n_e, t0, nv, first, last, wid == 0, lane);
        }
      }
      if (active) {
        __syncwarp();
        uint4* row = tile_row(tile, lane);  // carry: the block's last 32 bytes
        row[0] = row[8];
        row[1] = row[9];
        __syncwarp();
      }
      if (real && fb + 1 >= fb1) break;
    }
  }
  cp_async_wait<0>();
}

// Token blocks per unit for a launch over total_blocks blocks and ngroups
// feature groups on `wave` resident CTAs: the longest run up to kColRunMax
// whose units fill whole waves (k waves: at most k * wave units, the last
// wave nearly full), for the smallest such k.  A last wave of a few units
// would otherwise run alone on an idle GPU: at 616 units on 304 resident
// CTAs, eight units made a third wave.  Never below kColRunMin.
int64_t col_run_blocks(int64_t total_blocks, int64_t ngroups, int64_t wave) {
  for (int64_t k = 1; k <= 4096; ++k) {
    const int64_t nruns = k * wave / ngroups;
    if (nruns < 1) continue;
    const int64_t r = (total_blocks + nruns - 1) / nruns;
    if (r <= kColRunMax) return r < kColRunMin ? kColRunMin : r;
  }
  return kColRunMax;
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

fp4_status fp4_to_fp8_col_runs(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                               const int64_t* seg_row_off, const int64_t* seg_scale_off,
                               int32_t num_segments, int64_t total_rows, int64_t total_blocks,
                               int32_t run_blocks, uint8_t* fp8_t, float* fp8_t_scales,
                               void* stream) {
  if (cols < 0 || cols % 128 != 0 || num_segments < 0 || total_rows < 0 || total_blocks < 0 ||
      run_blocks < 0 || run_blocks > kColRunLimit)
    return FP4_ERR_SHAPE;
  if (total_blocks > total_rows / 128 + num_segments || total_blocks >= ((int64_t)1 << 31))
    return FP4_ERR_SHAPE;
  if (!seg_row_off || !seg_scale_off) return FP4_ERR_NULL;
  const int64_t ntiles = total_blocks * (cols / 128);
  if (ntiles > 0 && (!packed || !scales || !fp8_t || !fp8_t_scales)) return FP4_ERR_NULL;
  if (!aligned(packed, 32) || !aligned(scales, 4) || !aligned(fp8_t_scales, 4) ||
      !aligned(seg_row_off, 8) || !aligned(seg_scale_off, 8))
    return FP4_ERR_ALIGN;
  if (ntiles == 0 || num_segments == 0) return FP4_OK;
  if (!allow_dynamic_smem<fp4_to_fp8_col_kernel<true>>(kColSmem) ||
      !allow_dynamic_smem<fp4_to_fp8_col_kernel<false>>(kColSmem))
    return FP4_ERR_CUDA;
  // one CTA per (run of token blocks, group of kColGroup 32-feature blocks)
  const int64_t ngroups = (cols / 32 + kColGroup - 1) / kColGroup;
  const int64_t run =
      run_blocks > 0
          ? run_blocks
          : col_run_blocks(total_blocks, ngroups,
                           wave_ctas<fp4_to_fp8_col_kernel<true>>(kColThreads, kColSmem));
  const int64_t nunits = (total_blocks + run - 1) / run * ngroups;
  if (num_segments + 1 <= kSegTab)
    return launch<fp4_to_fp8_col_kernel<true>>(nunits * kColThreads, kColThreads, kColSmem,
                                               as_stream(stream), packed, scales, cols,
                                               seg_row_off, seg_scale_off, num_segments,
                                               total_blocks, run, nunits, fp8_t, fp8_t_scales);
  return launch<fp4_to_fp8_col_kernel<false>>(nunits * kColThreads, kColThreads, kColSmem,
                                              as_stream(stream), packed, scales, cols,
                                              seg_row_off, seg_scale_off, num_segments,
                                              total_blocks, run, nunits, fp8_t, fp8_t_scales);
}

fp4_status fp4_to_fp8_col(const uint8_t* packed, const uint8_t* scales, int64_t cols,
                          const int64_t* seg_row_off, const int64_t* seg_scale_off,
                          int32_t num_segments, int64_t total_rows, int64_t total_blocks,
                          uint8_t* fp8_t, float* fp8_t_scales, void* stream) {
  return fp4_to_fp8_col_runs(packed, scales, cols, seg_row_off, seg_scale_off, num_segments,
                             total_rows, total_blocks, 0, fp8_t, fp8_t_scales, stream);
}

}  // extern "C"
