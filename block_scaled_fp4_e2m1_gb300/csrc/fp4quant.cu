// fp4quant.cu -- FP4Quant group encode / decode.
//
// [FP4Quant] "Why four bits need more than rounding": each contiguous group
// gets an RMS scale, then a normalized Walsh-Hadamard transform made of
// additions and subtractions, then an absmax scale into the E2M1 range; both
// scales travel with the codes.  "Making compression cheap enough to help":
// the transform's early stages stay inside a thread, the stages that span
// threads exchange values through on-chip memory, codes are packed two per
// byte in registers, and the receiver unpacks, dequantizes and runs the
// inverse transform.
//
// Layout.  A group of G elements spans L = G/32 consecutive lanes (2, 4 or
// 8), never leaving its warp: no CTA barrier.  The transform's stages run in
// the natural (Sylvester) order h = 1, 2, ..., G/2, which the CPU oracle
// follows, in two phases:
//   - phase 1: lane l holds the 32 consecutive elements 32 l .. 32 l + 31 of
//     the group (staged through shared memory by cp.async), so the sum of
//     squares and the stages h = 1 .. 16 are in-thread;
//   - a transpose through a warp-private shared-memory tile: lane l then
//     holds, for every lane i of its group, the 32/L consecutive elements
//     32 i + l (32/L) .. of i's chunk; the tile's 16-byte units are placed
//     so that the eight lanes of a quarter-warp touch eight different bank
//     groups on every 128-bit store and load, at addresses that are a
//     per-lane base plus a constant;
//   - phase 2: the stages h = 32 .. G/2 pair elements of chunks i and
//     i xor (h/32), now in the same thread.
// Each stage is one correctly rounded add and subtract per pair, two pairs
// per packed f32x2 instruction.  The codes (encode) and the values (decode)
// leave phase 2 as one store per source chunk of 32/L codes or values, the
// L lanes of a group covering each chunk's row contiguously.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"
#include "rn_math.cuh"

namespace fp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kE = 32;                      // elements per lane

template <int G>
__device__ __forceinline__ float wht_norm() {
  // RN(1/sqrt(G)): 1/8, RN(sqrt(2)/16) = 0x3DB504F3, 1/16
  return G == 64 ? 0.125f : (G == 256 ? 0.0625f : __uint_as_float(0x3DB504F3u));
}

__device__ __forceinline__ F2 splat(float v) { return F2{v, v}; }

// 32 elements of a lane as 16 packed pairs.  Phase 1: p[t] holds elements
// 2t, 2t + 1 of the lane's chunk.  Phase 2: p[i * B/2 + t] holds elements
// 2t, 2t + 1 of the lane's block of chunk i of the group (B = 32/L).
struct Row32 {
  F2 p[16];
};

// No packed product feeds a packed addition: the compiler may fuse the two
// into one packed fma (one rounding instead of two), which would break the
// exact operation order.  A packed product may feed the scalar addition of
// its own two halves (stage h = 1), which no fma can absorb.

// Stages h = 1 .. 16 of the transform, inside the thread (phase 1).
__device__ __forceinline__ void wht_in_thread(Row32& y) {
#pragma unroll
  for (int t = 0; t < 16; ++t) {  // h = 1: the two halves of each pair
    const float a = y.p[t].x, b = y.p[t].y;
    y.p[t] = F2{__fadd_rn(a, b), __fsub_rn(a, b)};
  }
#pragma unroll
  for (int hp = 1; hp < 16; hp <<= 1) {  // h = 2 hp
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      if (t & hp) continue;
      const F2 a = y.p[t], b = y.p[t + hp];
      y.p[t] = add2(a, b);
      y.p[t + hp] = sub2(a, b);
    }
  }
}

// Stages h = 32 .. G/2 on the phase-2 layout: chunk index bit m of the
// group is the register block index bit m.
template <int G>
__device__ __forceinline__ void wht_across_chunks(Row32& y) {
  constexpr int L = G / kE, BP = 16 / L;  // pairs per chunk block
#pragma unroll
  for (int m = 1; m < L; m <<= 1) {
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if (i & m) continue;
#pragma unroll
      for (int t = 0; t < BP; ++t) {
        const F2 a = y.p[i * BP + t], b = y.p[(i + m) * BP + t];
        y.p[i * BP + t] = add2(a, b);
        y.p[(i + m) * BP + t] = sub2(a, b);
      }
    }
  }
}

// The phase-1 -> phase-2 transpose through the warp's 4.5 KB shared tile.
// Group g owns the 9 L units from unit 9 L g.  Lane l of the group writes its
// block k (elements k B .. k B + B - 1), in S = 8/L 16-byte halves h, to unit
// l + L h + 9 k of the group's region, and reads lane i's block l half h
// from unit i + L h + 9 l.  Both sides are a per-lane base plus a constant,
// so no address is computed per access.  l + L h covers 0 .. 7 once, so the
// blocks (9 units apart) do not overlap; and since 9 L = L and 9 = 1 mod 8,
// the eight lanes of a quarter-warp (S groups of L lanes) touch eight
// different units mod 8 on every store and load: no bank conflict.
template <int G>
struct TTile {
  static constexpr int L = G / kE;
  static constexpr int kBytes = 16 * 32 * 9;  // per warp: 32/L regions of 9 L units
};

template <int G>
__device__ __forceinline__ void transpose_to_blocks(Row32& y, float4* tile, int lane) {
  constexpr int L = G / kE, B = kE / L, S = 8 / L;
  const int g = lane / L, l = lane % L;
  float4* const st = tile + 9 * L * g + l;
  const float4* const ld = tile + 9 * L * g + 9 * l;
#pragma unroll
  for (int k = 0; k < L; ++k) {
#pragma unroll
    for (int h = 0; h < S; ++h) {
      const F2 a = y.p[k * B / 2 + 2 * h], b = y.p[k * B / 2 + 2 * h + 1];
      st[L * h + 9 * k] = make_float4(a.x, a.y, b.x, b.y);
    }
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < L; ++i) {
#pragma unroll
    for (int h = 0; h < S; ++h) {
      const float4 v = ld[i + L * h];
      y.p[i * B / 2 + 2 * h] = F2{v.x, v.y};
      y.p[i * B / 2 + 2 * h + 1] = F2{v.z, v.w};
    }
  }
  __syncwarp();
}

// max(0, |v|) over a lane's 32 values, as a tree of three-input maxima (16
// instructions, 4 deep) rather than a chain.
__device__ __forceinline__ float absmax32(const Row32& y) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[2 * i] = y.p[i].x;
    v[2 * i + 1] = y.p[i].y;
  }
  float a[10];
#pragma unroll
  for (int k = 0; k < 10; ++k) a[k] = max3_abs(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  const float b0 = max3(a[0], a[1], a[2]), b1 = max3(a[3], a[4], a[5]);
  const float b2 = max3(a[6], a[7], a[8]), b3 = max3_abs(a[9], v[30], v[31]);
  return max3(max3(b0, b1, b2), b3, 0.0f);
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int m = 1; m < G / kE; m <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int m = 1; m < G / kE; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

// Per-warp staging ring in shared memory for a kernel's input.  A tile is
// what the warp's 32 lanes consume in one loop step, P 16-byte pieces per
// lane, contiguous in global memory (lane c's pieces at 16 (P c + q)).  The
// warp copies a tile with cp.async, piece 32 k + lane in instruction k, so
// each copy instruction reads 512 contiguous bytes; tiles are copied NS - 1
// steps ahead of their use, so several tiles per warp are in flight without
// holding registers.  In shared memory lane c's piece q sits at unit
// P c + (q xor sw(c)), sw(c) = (c / (8/P)) mod P: the eight lanes of a
// quarter-warp then touch eight different 16-byte units mod 128 bytes, for
// the copies and for each lane's 128-bit reads of its own pieces.
template <int P>
__device__ __forceinline__ int ring_unit(int c, int q) {
  return P * c + (q ^ ((c / (8 / P)) & (P - 1)));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 4 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async16_all(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Byte offset in a slot of piece 32 k + lane: 512 (k - k mod M) plus a lane
// offset that depends on k only through k mod M (M = 2 for P = 8, else 1),
// so every copy of a tile is one per-lane base plus a constant.
template <int P>
__device__ __forceinline__ uint32_t ring_piece_off(int lane, int k) {
  constexpr int M = P == 8 ? 2 : 1;
  const int p = 32 * (k % M) + lane;
  return 16u * (uint32_t)ring_unit<P>(p / P, p % P) + 512u * (uint32_t)(k - k % M);
}

// Copies a whole tile (lane's pieces at src_lane + 512 k) into the slot at
// byte address dst.
template <int P>
__device__ __forceinline__ void ring_copy_full(uint32_t dst, const uint8_t* src_lane, int lane) {
#pragma unroll
  for (int k = 0; k < P; ++k) cp_async16_all(dst + ring_piece_off<P>(lane, k), src_lane + 512 * k);
}

// Copies the tile at src (valid: its first `valid` bytes exist, a multiple
// of 16; the rest is zero-filled without reading) into the slot at byte
// address dst.
template <int P>
__device__ __forceinline__ void ring_copy(uint32_t dst, const uint8_t* src, int64_t valid,
                                          int lane) {
#pragma unroll
  for (int k = 0; k < P; ++k) {
    const int p = 32 * k + lane;
    const bool ok = 16 * (int64_t)p < valid;
    cp_async16(dst + ring_piece_off<P>(lane, k), ok ? src + 16 * p : src, ok);
  }
}

// Lane's P pieces of the tile in the slot at byte address slot (64-byte
// aligned): piece q at (slot + 16 P lane + 16 sw) xor 16 q.
template <int P>
__device__ __forceinline__ void ring_read(uint32_t slot, int lane, uint4 v[P]) {
  const uint32_t a = slot + 16u * (uint32_t)ring_unit<P>(lane, 0);
#pragma unroll
  for (int q = 0; q < P; ++q)
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[q].x), "=r"(v[q].y), "=r"(v[q].z), "=r"(v[q].w)
                 : "r"(a ^ (16u * (uint32_t)q))
                 : "memory");
}

__device__ __forceinline__ float bf16_lo_(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// A lane's 32 input elements from its P = 4 (bf16) or 8 (fp32) pieces.
template <bool kBF16>
__device__ __forceinline__ void unpack_chunk(const uint4* v, Row32& y) {
  if (kBF16) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) y.p[4 * q + i] = F2{bf16_lo_(w[i]), bf16_hi_(w[i])};
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      y.p[2 * q] = F2{__uint_as_float(v[q].x), __uint_as_float(v[q].y)};
      y.p[2 * q + 1] = F2{__uint_as_float(v[q].z), __uint_as_float(v[q].w)};
    }
  }
}

// Stores the B codes of each source chunk of the group: B = 4 -> 2 bytes,
// 8 -> 4 bytes, 16 -> 8 bytes at byte l B / 2 of the chunk's 16-byte row.
template <int B>
__device__ __forceinline__ void store_codes(uint8_t* row, int l, const uint32_t* w) {
  if (B == 4) {
    *reinterpret_cast<uint16_t*>(row + 2 * l) = (uint16_t)w[0];
  } else if (B == 8) {
    *reinterpret_cast<uint32_t*>(row + 4 * l) = w[0];
  } else {
    *reinterpret_cast<uint2*>(row + 8 * l) = make_uint2(w[0], w[1]);
  }
}

// Encodes the group chunk set this warp holds (tile t: lane's chunk
// 32 t + lane, valid when inside the tensor) and stores codes and scales.
// Lanes past the end compute on zeros and store nothing (the chunk count is
// a multiple of L, so a group is either entirely inside or entirely past the
// end).
template <int G>
__device__ __forceinline__ void encode_chunk(Row32& y, int t, bool valid, int lane, float4* tile,
                                             uint8_t* __restrict__ packed,
                                             float* __restrict__ s1_out,
                                             float* __restrict__ s2_out) {
  constexpr int L = G / kE, B = kE / L;
  // RMS scale: the pairwise tree over adjacent squares, levels 2-5 two sums
  // per instruction (the halves 0..15 | 16..31 side by side)
  F2 sq[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const F2 a = mul2(y.p[i], y.p[i]), b = mul2(y.p[8 + i], y.p[8 + i]);
    sq[i] = F2{__fadd_rn(a.x, a.y), __fadd_rn(b.x, b.y)};
  }
#pragma unroll
  for (int w = 8; w > 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w / 2; ++i) sq[i] = add2(sq[2 * i], sq[2 * i + 1]);
  }
  const float ss = group_sum<G>(__fadd_rn(sq[0].x, sq[0].y));
  const float rms = sqrt_rn(__fmul_rn(ss, 1.0f / (float)G));
  const float inv1 = rms == 0.0f ? 0.0f : rcp_rn(rms);
#pragma unroll
  for (int i = 0; i < 16; ++i) y.p[i] = mul2(y.p[i], splat(inv1));
  // transform: stages 1..16, transpose, stages 32..G/2, normalization
  wht_in_thread(y);
  transpose_to_blocks<G>(y, tile, lane);
  wht_across_chunks<G>(y);
  // normalization and absmax scale into [-6, 6].  z = RN(w c) and
  // max|z| = RN(max|w| c) (RN is monotone).  For G = 64 and 256, c is a
  // power of two: when 2^-20 <= max|z| <= 2^100, RN(z inv2) = RN(w (c inv2))
  // for every element (c inv2 is exact; where w c is normal, z = w c
  // exactly; where it is subnormal, both products are below 2^-100 and
  // round to a zero code of w's sign), so the two scalings fold into one.
  const float c = wht_norm<G>();
  const float zmax = __fmul_rn(group_max<G>(absmax32(y)), c);
  const float sc2 = div6_rn(zmax);
  const float inv2 = sc2 == 0.0f ? 0.0f : rcp_rn(sc2);
  if (G != 128 && zmax >= 0x1p-20f && zmax <= 0x1p100f) {
    const F2 m = splat(__fmul_rn(inv2, c));
#pragma unroll
    for (int i = 0; i < 16; ++i) y.p[i] = mul2(y.p[i], m);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) y.p[i] = mul2(mul2(y.p[i], splat(c)), splat(inv2));
  }
  if (!valid) return;
  const int l = lane % L;
  // the group's first chunk row
  uint8_t* const rows = packed + 16 * ((int64_t)t * 32 + (lane - l));
  if (B == 4) {
    // two source chunks' 4 codes per conversion word, stored as halves
#pragma unroll
    for (int i = 0; i < L; i += 2) {
      const F2* q = y.p + i * 2;
      const uint32_t w = cvt_e2m1x8(q[0].x, q[0].y, q[1].x, q[1].y, q[2].x, q[2].y, q[3].x,
                                    q[3].y);
      *reinterpret_cast<uint16_t*>(rows + 16 * i + 2 * l) = (uint16_t)w;
      *reinterpret_cast<uint16_t*>(rows + 16 * (i + 1) + 2 * l) = (uint16_t)(w >> 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < L; ++i) {
      const F2* q = y.p + i * (B / 2);
      uint32_t w[2];
#pragma unroll
      for (int k = 0; k < B / 8; ++k)
        w[k] = cvt_e2m1x8(q[4 * k].x, q[4 * k].y, q[4 * k + 1].x, q[4 * k + 1].y,
                          q[4 * k + 2].x, q[4 * k + 2].y, q[4 * k + 3].x, q[4 * k + 3].y);
      store_codes<B>(rows + 16 * i, l, w);
    }
  }
  if (l == 0) {
    const int64_t gi = (int64_t)t * (32 / L) + lane / L;
    s1_out[gi] = rms;
    s2_out[gi] = sc2;
  }
}

// Input pieces per lane and the shared memory of the encode kernels: one
// staging slot per warp plus its transpose tile.  (bf16: 6.5 KB per warp,
// four CTAs of 256 threads per SM at 64 registers; fp32: 8.5 KB per warp,
// two CTAs.)
template <int G, bool kBF16>
struct EncRing {
  static constexpr int P = kBF16 ? 4 : 8;            // 64 or 128 bytes per lane
  static constexpr int kSlot = 32 * 16 * P;          // bytes per tile
  static constexpr size_t kSmem = (size_t)kWarps * (kSlot + TTile<G>::kBytes);
};

// The loop walks 32-chunk tiles, one per warp per grid-stride step, and is
// warp-uniform so that every lane takes part in the exchanges.  Each warp
// stages its next tile into its one shared slot as soon as it has read the
// current tile out of it (one cp.async group per tile, committed even when
// empty), so the copy runs under the current tile's arithmetic without
// holding registers.  Tile indices are 32-bit (the entry point admits fewer
// than 2^35 chunks).
template <int G, bool kBF16>
__global__ void __launch_bounds__(kThreads, kBF16 ? 4 : 2)
    encode_kernel(const void* __restrict__ x, int64_t nchunks, uint8_t* __restrict__ packed,
                  float* __restrict__ s1_out, float* __restrict__ s2_out) {
  using R = EncRing<G, kBF16>;
  constexpr int P = R::P;
  extern __shared__ __align__(128) uint8_t enc_smem[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t slot = (uint32_t)__cvta_generic_to_shared(enc_smem) + (uint32_t)(wid * R::kSlot);
  float4* const tile =
      reinterpret_cast<float4*>(enc_smem + kWarps * R::kSlot + wid * TTile<G>::kBytes);
  const int ntiles = (int)((nchunks + 31) >> 5), nfull = (int)(nchunks >> 5);
  const int rem = (int)(nchunks & 31);
  const int tstride = (int)gridDim.x * kWarps;
  const int64_t step = (int64_t)tstride * R::kSlot;  // input bytes between a warp's tiles
  int t = (int)blockIdx.x * kWarps + wid;
  const uint8_t* src = static_cast<const uint8_t*>(x) + (int64_t)t * R::kSlot;
  auto stage = [&](int tt, const uint8_t* s) {
    if (tt < nfull)
      ring_copy_full<P>(slot, s + 16 * lane, lane);
    else if (tt < ntiles)
      ring_copy<P>(slot, s, (nchunks - 32 * (int64_t)tt) * (16 * P), lane);
    cp_async_commit();
  };
  stage(t, src);
  for (; t < ntiles; t += tstride, src += step) {
    cp_async_wait<0>();
    __syncwarp();
    uint4 v[P];
    ring_read<P>(slot, lane, v);
    __syncwarp();  // every lane's reads of the slot before its next copy
    stage(t + tstride, src + step);
    Row32 y;
    unpack_chunk<kBF16>(v, y);
    encode_chunk<G>(y, t, t < nfull || lane < rem, lane, tile, packed, s1_out, s2_out);
  }
  cp_async_wait<0>();
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Staged tiles of the decode kernels: per tile the 32 chunks' codes (16
// bytes per lane) and the s1, s2 of its 32/L groups.
template <int G>
struct DecRing {
  static constexpr int L = G / kE, NG = 32 / L;
  static constexpr int NS = 4;                       // tiles per warp ring
  static constexpr int kSlot = 512 + 8 * NG;         // bytes per tile (multiple of 16)
  static constexpr size_t kSmem = (size_t)kWarps * (NS * kSlot + TTile<G>::kBytes);
};

// Stores the B values of each source chunk: bf16 B = 4, 8, 16 -> 8, 16, 32
// bytes; fp32 -> 16, 32, 64 bytes, at element l B of the chunk's row.
template <int B, bool kBF16Out>
__device__ __forceinline__ void store_values(void* out, int64_t chunk, int l, const F2* q) {
  if (kBF16Out) {
    uint16_t* o = static_cast<uint16_t*>(out) + kE * chunk + B * l;
    uint32_t w[B / 2];
#pragma unroll
    for (int t = 0; t < B / 2; ++t) w[t] = pack_bf16x2(q[t].x, q[t].y);
    if (B == 4) {
      *reinterpret_cast<uint2*>(o) = make_uint2(w[0], w[1]);
    } else if (B == 8) {
      *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      U32x8 v;
#pragma unroll
      for (int t = 0; t < 8; ++t) v.w[t] = w[t];
      st_v8(o, v);
    }
  } else {
    float* o = static_cast<float*>(out) + kE * chunk + B * l;
    if (B == 4) {
      *reinterpret_cast<float4*>(o) = make_float4(q[0].x, q[0].y, q[1].x, q[1].y);
    } else {
#pragma unroll
      for (int k = 0; k < B / 8; ++k) {
        U32x8 v;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          v.w[2 * t] = __float_as_uint(q[4 * k + t].x);
          v.w[2 * t + 1] = __float_as_uint(q[4 * k + t].y);
        }
        st_v8(o + 8 * k, v);
      }
    }
  }
}

// Tiles are staged NS - 1 loop steps ahead in the warp's ring, as in the
// encode kernels; tile indices are 32-bit likewise.  The bf16-output
// kernels for G = 128 and 256 are held to 64 registers (four CTAs per SM);
// for G = 64 three CTAs at 71 registers measured faster.
template <int G, bool kBF16Out>
__global__ void __launch_bounds__(kThreads, (kBF16Out && G != 64) ? 4 : 1)
    decode_kernel(const uint8_t* __restrict__ packed, const float* __restrict__ s1_in,
                  const float* __restrict__ s2_in, int64_t nchunks, void* __restrict__ out) {
  using R = DecRing<G>;
  constexpr int L = G / kE, B = kE / L, NG = R::NG, NS = R::NS;
  extern __shared__ __align__(128) uint8_t dec_smem[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int l = lane % L;
  const uint32_t ring =
      (uint32_t)__cvta_generic_to_shared(dec_smem) + (uint32_t)(wid * NS * R::kSlot);
  float4* const tile =
      reinterpret_cast<float4*>(dec_smem + kWarps * NS * R::kSlot + wid * TTile<G>::kBytes);
  const int ntiles = (int)((nchunks + 31) >> 5), nfull = (int)(nchunks >> 5);
  const int rem = (int)(nchunks & 31);
  const int64_t ngroups = nchunks / L;
  const int tstride = (int)gridDim.x * kWarps;
  int t = (int)blockIdx.x * kWarps + wid;
  // lanes 0 .. NG-1 stage the tile's s1 words, lanes NG .. 2 NG-1 its s2 words
  const float* const ssrc = (lane < NG ? s1_in : s2_in) + (lane % NG);
  auto stage = [&](int tt, int slot) {
    const uint32_t dst = ring + (uint32_t)(slot * R::kSlot);
    if (tt < nfull) {
      cp_async16_all(dst + 16u * lane, packed + 512 * (int64_t)tt + 16 * lane);
      if (lane < 2 * NG) cp_async4(dst + 512u + 4u * lane, ssrc + (int64_t)tt * NG, true);
    } else if (tt < ntiles) {
      const int64_t t0 = 32 * (int64_t)tt;
      ring_copy<1>(dst, packed + 16 * t0, (nchunks - t0) * 16, lane);
      const int64_t gi = t0 / L + (lane % NG);
      const bool ok = lane < 2 * NG && gi < ngroups;
      const float* src = lane < NG ? s1_in : s2_in;
      if (lane < 2 * NG) cp_async4(dst + 512u + 4u * lane, ok ? src + gi : src, ok);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int k = 0; k < NS - 1; ++k) stage(t + k * tstride, k);
  for (int it = 0; t < ntiles; ++it, t += tstride) {
    stage(t + (NS - 1) * tstride, (it + NS - 1) % NS);
    cp_async_wait<NS - 1>();
    __syncwarp();
    const bool valid = t < nfull || lane < rem;
    const uint32_t slot = ring + (uint32_t)((it % NS) * R::kSlot);
    uint4 pk[1];
    ring_read<1>(slot, lane, pk);
    const float sc1 = ld_shared_f32(slot + 512u + 4u * (lane / L));
    const float sc2 = ld_shared_f32(slot + 512u + 4u * (NG + lane / L));
    Row32 z;
    const uint32_t words[4] = {pk[0].x, pk[0].y, pk[0].z, pk[0].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v[8];
      e2m1x8_to_f32(words[k], v);
#pragma unroll
      for (int i = 0; i < 4; ++i) z.p[4 * k + i] = mul2(F2{v[2 * i], v[2 * i + 1]}, splat(sc2));
    }
    wht_in_thread(z);
    transpose_to_blocks<G>(z, tile, lane);
    wht_across_chunks<G>(z);
    // normalization, then x' = y' s1 with the group's s1 (every lane of a
    // group holds it).  For G = 64 and 256, c is a power of two; when
    // s2 = 0 or |s2| >= 2^-60 every nonzero transform output w is a multiple
    // of 2^-84 (the values z are RN(v s2) >= 2^-61 in magnitude, and sums of
    // multiples of 2^-84 stay multiples of it), so w c is exact, and when
    // s1 = 0 or |s1| >= 2^-120 so is c s1: then RN(RN(w c) s1) = RN(w (c s1))
    // and one scaling does both.
    const float c = wht_norm<G>();
    const bool fold_ok = (sc2 == 0.0f || fabsf(sc2) >= 0x1p-60f) &&
                         (sc1 == 0.0f || fabsf(sc1) >= 0x1p-120f);
    if (G != 128 && __all_sync(0xFFFFFFFFu, fold_ok)) {
      const F2 m = splat(__fmul_rn(c, sc1));
#pragma unroll
      for (int i = 0; i < 16; ++i) z.p[i] = mul2(z.p[i], m);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) z.p[i] = mul2(mul2(z.p[i], splat(c)), splat(sc1));
    }
    if (valid) {
#pragma unroll
      for (int i = 0; i < L; ++i)
        store_values<B, kBF16Out>(out, (int64_t)t * 32 + (lane - l) + i, l, z.p + i * (B / 2));
    }
  }
  cp_async_wait<0>();
}

template <int G, bool kBF16>
fp4_status launch_encode_t(const void* x, int64_t nchunks, uint8_t* packed, float* s1, float* s2,
                           cudaStream_t s) {
  constexpr size_t smem = EncRing<G, kBF16>::kSmem;
  if (!allow_dynamic_smem<encode_kernel<G, kBF16>>(smem)) return FP4_ERR_CUDA;
  return launch<encode_kernel<G, kBF16>>(nchunks, kThreads, smem, s, x, nchunks, packed, s1, s2);
}

template <int G>
fp4_status launch_encode(const void* x, int dtype, int64_t nchunks, uint8_t* packed, float* s1,
                         float* s2, cudaStream_t s) {
  if (dtype == FP4_BF16) return launch_encode_t<G, true>(x, nchunks, packed, s1, s2, s);
  return launch_encode_t<G, false>(x, nchunks, packed, s1, s2, s);
}

template <int G, bool kBF16Out>
fp4_status launch_decode_t(const uint8_t* packed, const float* s1, const float* s2,
                           int64_t nchunks, void* y, cudaStream_t s) {
  constexpr size_t smem = DecRing<G>::kSmem;
  if (!allow_dynamic_smem<decode_kernel<G, kBF16Out>>(smem)) return FP4_ERR_CUDA;
  return launch<decode_kernel<G, kBF16Out>>(nchunks, kThreads, smem, s, packed, s1, s2, nchunks,
                                            y);
}

template <int G>
fp4_status launch_decode(const uint8_t* packed, const float* s1, const float* s2, int64_t nchunks,
                         void* y, int dtype, cudaStream_t s) {
  if (dtype == FP4_BF16) return launch_decode_t<G, true>(packed, s1, s2, nchunks, y, s);
  return launch_decode_t<G, false>(packed, s1, s2, nchunks, y, s);
}

bool group_ok(int g) { return g == 64 || g == 128 || g == 256; }

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

fp4_status fp4quant_encode(const void* x, int dtype, int64_t rows, int64_t cols, int group,
                           uint8_t* packed, float* s1, float* s2, void* stream) {
  if (!dtype_ok(dtype)) return FP4_ERR_DTYPE;
  if (!group_ok(group)) return FP4_ERR_ARG;
  if (rows < 0 || cols < 0 || cols % group != 0) return FP4_ERR_SHAPE;
  if (cols > 0 && rows > ((int64_t)1 << 40) / cols) return FP4_ERR_SHAPE;
  const int64_t nchunks = rows * cols / kE;
  if (nchunks > 0 && (!x || !packed || !s1 || !s2)) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(packed, 16) || !aligned(s1, 4) || !aligned(s2, 4))
    return FP4_ERR_ALIGN;
  if (nchunks == 0) return FP4_OK;
  cudaStream_t s = as_stream(stream);
  if (group == 64) return launch_encode<64>(x, dtype, nchunks, packed, s1, s2, s);
  if (group == 128) return launch_encode<128>(x, dtype, nchunks, packed, s1, s2, s);
  return launch_encode<256>(x, dtype, nchunks, packed, s1, s2, s);
}

fp4_status fp4quant_decode(const uint8_t* packed, const float* s1, const float* s2, int64_t rows,
                           int64_t cols, int group, void* y, int out_dtype, void* stream) {
  if (!dtype_ok(out_dtype)) return FP4_ERR_DTYPE;
  if (!group_ok(group)) return FP4_ERR_ARG;
  if (rows < 0 || cols < 0 || cols % group != 0) return FP4_ERR_SHAPE;
  if (cols > 0 && rows > ((int64_t)1 << 40) / cols) return FP4_ERR_SHAPE;
  const int64_t nchunks = rows * cols / kE;
  if (nchunks > 0 && (!y || !packed || !s1 || !s2)) return FP4_ERR_NULL;
  if (!aligned(y, 32) || !aligned(packed, 16) || !aligned(s1, 4) || !aligned(s2, 4))
    return FP4_ERR_ALIGN;
  if (nchunks == 0) return FP4_OK;
  cudaStream_t s = as_stream(stream);
  if (group == 64) return launch_decode<64>(packed, s1, s2, nchunks, y, out_dtype, s);
  if (group == 128) return launch_decode<128>(packed, s1, s2, nchunks, y, out_dtype, s);
  return launch_decode<256>(packed, s1, s2, nchunks, y, out_dtype, s);
}

}  // extern "C"
