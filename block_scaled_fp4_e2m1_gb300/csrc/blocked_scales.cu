// blocked_scales.cu -- block scales between the linear [rows, cols] layout
// the quantizers write and the blocked (swizzled) layout Blackwell
// block-scaled tensor-core matmuls read.
//
// [fp4-train] "Scope": the NVFP4 tensor-core matmul swizzles its e4m3 block
// scales into the layout torch._scaled_mm consumes.  The layout (common.cuh):
// zero padding to whole tiles of 128 rows x 4 scale columns, tiles in
// row-major order, 512 bytes each, scale (r, c) of a tile at byte
// 16 (r mod 32) + 4 floor(r / 32) + c.  It is the same for NVFP4 (e4m3, one
// per 16 elements) and MXFP4 (UE8M0, one per 32) scales: bytes are moved,
// never interpreted.
//
// Layout of the work: one CTA unit is 128 rows x up to 32 column tiles (128
// scale columns).  Its blocked bytes are one contiguous run of up to 16 KB,
// and its linear bytes are 128 row segments of up to 128 B.  The unit goes
// through shared memory ([128][132] bytes: a row pitch of 33 words keeps
// both the row-segment side and the 16-byte-line side free of bank
// conflicts), so both HBM sides are read and written in full 128-byte
// lines.  HBM-bound: rows * cols bytes on one side, the padded size on the
// other.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"

namespace fp4 {
namespace {

constexpr int kTThreads = 256;
constexpr int kUnitTiles = 32;           // column tiles per unit
constexpr int kUnitCols = 4 * kUnitTiles;  // scale columns per unit
constexpr int kPitch = kUnitCols + 4;    // shared row pitch in bytes

struct Geometry {
  int64_t rows, cols;     // linear scale matrix
  int64_t col_tiles;      // ceil(cols / 4)
  int64_t units_per_row;  // ceil(col_tiles / kUnitTiles)
  int64_t units;          // ceil(rows / 128) * units_per_row
};

// The unit's place: first row r0, first scale column c0, tiles in the unit,
// valid rows and valid columns (the rest is padding).
struct Unit {
  int64_t r0, c0, out0;  // out0: byte offset of the unit's first tile
  int ntiles, vrows, vcols;
};

__device__ __forceinline__ Unit unit_at(const Geometry& g, int64_t u) {
  Unit t;
  const int64_t rt = u / g.units_per_row, ch = u - rt * g.units_per_row;
  t.r0 = rt * 128;
  t.c0 = ch * kUnitCols;
  t.out0 = (rt * g.col_tiles + ch * kUnitTiles) << 9;
  t.ntiles = (int)min((int64_t)kUnitTiles, g.col_tiles - ch * kUnitTiles);
  t.vrows = (int)min((int64_t)128, g.rows - t.r0);
  t.vcols = (int)min((int64_t)(4 * t.ntiles), g.cols - t.c0);
  return t;
}

// Row segment element j (kVec bytes) of linear row i in the unit <-> shared
// memory.  With cols % kVec == 0 and a kVec-aligned base every access is
// aligned: units start at a multiple of 128 columns.
template <int kVec>
__device__ __forceinline__ void seg_to_smem(const uint8_t* src, uint8_t* dst) {
  if (kVec == 16) {
    const uint4 q = ld_stream_v4(src);
    uint32_t* d = reinterpret_cast<uint32_t*>(dst);
    d[0] = q.x;
    d[1] = q.y;
    d[2] = q.z;
    d[3] = q.w;
  } else if (kVec == 4) {
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
  } else {
    *dst = *src;
  }
}

template <int kVec>
__device__ __forceinline__ void smem_to_seg(const uint8_t* src, uint8_t* dst) {
  if (kVec == 16) {
    const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
    *reinterpret_cast<uint4*>(dst) = make_uint4(s[0], s[1], s[2], s[3]);
  } else if (kVec == 4) {
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
  } else {
    *dst = *src;
  }
}

template <int kVec>
__device__ __forceinline__ void zero_seg(uint8_t* dst) {
  if (kVec == 1) {
    *dst = 0;
  } else {
#pragma unroll
    for (int k = 0; k < kVec / 4; ++k) reinterpret_cast<uint32_t*>(dst)[k] = 0u;
  }
}

// Linear -> blocked.  Every byte of the unit's blocked run is written:
// padding rows and columns come out of shared memory as zeros.
template <int kVec>
__global__ void __launch_bounds__(kTThreads)
    to_blocked_kernel(const uint8_t* __restrict__ in, Geometry g, uint8_t* __restrict__ out) {
  __shared__ __align__(16) uint8_t tile[128 * kPitch];
  constexpr int kPerRow = kUnitCols / kVec;
  for (int64_t u = blockIdx.x; u < g.units; u += gridDim.x) {
    const Unit t = unit_at(g, u);
    const int ncols = 4 * t.ntiles;
    for (int v = threadIdx.x; v < 128 * kPerRow; v += kTThreads) {
      const int i = v / kPerRow, j = (v - i * kPerRow) * kVec;
      if (j >= ncols) continue;
      uint8_t* dst = tile + i * kPitch + j;
      if (i < t.vrows && j < t.vcols)
        seg_to_smem<kVec>(in + (t.r0 + i) * g.cols + t.c0 + j, dst);
      else
        zero_seg<kVec>(dst);
    }
    __syncthreads();
    uint4* o = reinterpret_cast<uint4*>(out + t.out0);
    for (int w = threadIdx.x; w < 32 * t.ntiles; w += kTThreads) {
      const int tt = w >> 5, i = w & 31;
      const uint8_t* s = tile + i * kPitch + 4 * tt;
      uint4 q;
      q.x = *reinterpret_cast<const uint32_t*>(s);
      q.y = *reinterpret_cast<const uint32_t*>(s + 32 * kPitch);
      q.z = *reinterpret_cast<const uint32_t*>(s + 64 * kPitch);
      q.w = *reinterpret_cast<const uint32_t*>(s + 96 * kPitch);
      o[w] = q;
    }
    __syncthreads();
  }
}

// Blocked -> linear: the unit's blocked run into shared memory, then its
// valid rows and columns out.  Padding bytes are read and dropped.
template <int kVec>
__global__ void __launch_bounds__(kTThreads)
    from_blocked_kernel(const uint8_t* __restrict__ in, Geometry g, uint8_t* __restrict__ out) {
  __shared__ __align__(16) uint8_t tile[128 * kPitch];
  constexpr int kPerRow = kUnitCols / kVec;
  for (int64_t u = blockIdx.x; u < g.units; u += gridDim.x) {
    const Unit t = unit_at(g, u);
    const uint4* src = reinterpret_cast<const uint4*>(in + t.out0);
    for (int w = threadIdx.x; w < 32 * t.ntiles; w += kTThreads) {
      const int tt = w >> 5, i = w & 31;
      const uint4 q = ld_stream_v4(src + w);
      uint8_t* d = tile + i * kPitch + 4 * tt;
      *reinterpret_cast<uint32_t*>(d) = q.x;
      *reinterpret_cast<uint32_t*>(d + 32 * kPitch) = q.y;
      *reinterpret_cast<uint32_t*>(d + 64 * kPitch) = q.z;
      *reinterpret_cast<uint32_t*>(d + 96 * kPitch) = q.w;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < 128 * kPerRow; v += kTThreads) {
      const int i = v / kPerRow, j = (v - i * kPerRow) * kVec;
      if (i < t.vrows && j < t.vcols)
        smem_to_seg<kVec>(tile + i * kPitch + j, out + (t.r0 + i) * g.cols + t.c0 + j);
    }
    __syncthreads();
  }
}

Geometry geometry(int64_t rows, int64_t cols) {
  Geometry g;
  g.rows = rows;
  g.cols = cols;
  g.col_tiles = (cols + 3) / 4;
  g.units_per_row = (g.col_tiles + kUnitTiles - 1) / kUnitTiles;
  g.units = ((rows + 127) / 128) * g.units_per_row;
  return g;
}

// Widest access both the column count and the linear pointer allow.
int vec_width(const void* linear, int64_t cols) {
  if (cols % 16 == 0 && aligned(linear, 16)) return 16;
  if (cols % 4 == 0 && aligned(linear, 4)) return 4;
  return 1;
}

template <auto Kernel>
fp4_status launch_units(const Geometry& g, const uint8_t* in, uint8_t* out, cudaStream_t s) {
  static const int occ = occupancy(Kernel, kTThreads, 0);
  int64_t grid = (int64_t)sm_count() * occ;
  if (grid > g.units) grid = g.units;
  Kernel<<<(unsigned)grid, kTThreads, 0, s>>>(in, g, out);
  return after_launch();
}

bool blocked_shape_ok(int64_t rows, int64_t cols) {
  return rows >= 0 && cols >= 0 && rows < (INT64_C(1) << 40) && cols < (INT64_C(1) << 40) &&
         (cols == 0 || rows <= (INT64_C(1) << 44) / (cols + 3));
}

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

int64_t fp4_blocked_scales_size(int64_t rows, int64_t cols) {
  if (!blocked_shape_ok(rows, cols)) return -1;
  return ((rows + 127) / 128) * 128 * ((cols + 3) / 4) * 4;
}

fp4_status fp4_scales_to_blocked(const uint8_t* scales, int64_t rows, int64_t cols,
                                 uint8_t* blocked, void* stream) {
  if (!blocked_shape_ok(rows, cols)) return FP4_ERR_SHAPE;
  const Geometry g = geometry(rows, cols);
  if (g.units == 0) return FP4_OK;
  if (!scales || !blocked) return FP4_ERR_NULL;
  if (!aligned(blocked, 16)) return FP4_ERR_ALIGN;
  cudaStream_t s = as_stream(stream);
  switch (vec_width(scales, cols)) {
    case 16: return launch_units<to_blocked_kernel<16>>(g, scales, blocked, s);
    case 4: return launch_units<to_blocked_kernel<4>>(g, scales, blocked, s);
    default: return launch_units<to_blocked_kernel<1>>(g, scales, blocked, s);
  }
}

fp4_status fp4_scales_from_blocked(const uint8_t* blocked, int64_t rows, int64_t cols,
                                   uint8_t* scales, void* stream) {
  if (!blocked_shape_ok(rows, cols)) return FP4_ERR_SHAPE;
  const Geometry g = geometry(rows, cols);
  if (g.units == 0) return FP4_OK;
  if (!scales || !blocked) return FP4_ERR_NULL;
  if (!aligned(blocked, 16)) return FP4_ERR_ALIGN;
  cudaStream_t s = as_stream(stream);
  switch (vec_width(scales, cols)) {
    case 16: return launch_units<from_blocked_kernel<16>>(g, blocked, scales, s);
    case 4: return launch_units<from_blocked_kernel<4>>(g, blocked, scales, s);
    default: return launch_units<from_blocked_kernel<1>>(g, blocked, scales, s);
  }
}

}  // extern "C"
