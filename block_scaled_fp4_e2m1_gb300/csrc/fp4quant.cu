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
// The transform's stages run in the natural (Sylvester) order h = 1, 2,
// ..., G/2, which the CPU oracle follows; each stage is one correctly
// rounded add and subtract per pair, two pairs per packed f32x2
// instruction.  A group never leaves its warp: no CTA barrier.
//
// Encode layout: a lane holds whole chunk pairs of its group, 64 or 128
// elements (see the encode section below); G = 64 and 128 exchange nothing
// between lanes, G = 256 transposes once through a warp-private tile.
//
// Decode layout: a group spans L = G/32 consecutive lanes (2, 4 or 8), in
// two phases:
//   - phase 1: lane l holds the 32 consecutive elements 32 l .. 32 l + 31 of
//     the group (its codes staged through shared memory by cp.async), so
//     the stages h = 1 .. 16 are in-thread;
//   - a transpose through a warp-private shared-memory tile: lane l then
//     holds, for every lane i of its group, the 32/L consecutive elements
//     32 i + l (32/L) .. of i's chunk; the tile's 16-byte units are placed
//     so that the eight lanes of a quarter-warp touch eight different bank
//     groups on every 128-bit store and load, at addresses that are a
//     per-lane base plus a constant;
//   - phase 2: the stages h = 32 .. G/2 pair elements of chunks i and
//     i xor (h/32), now in the same thread.
// The values leave phase 2 as one store per source chunk of 32/L values,
// the L lanes of a group covering each chunk's row contiguously.
#include <cuda.h>
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
struct TTile {
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

// Per-warp staging ring in shared memory for a kernel's input.  A tile is
// what the warp's 32 lanes consume in one loop step, P 16-byte pieces per
// lane, contiguous in global memory (lane c's pieces at 16 (P c + q)).  The
// warp copies a tile with cp.async, piece 32 k + lane in instruction k, so
// each copy instruction reads 512 contiguous bytes; tiles are copied ahead of
// their use, so tiles are in flight without holding registers.  In shared
// memory lane c's piece q sits at unit P c + (q xor sw(c)), with
// sw(c) = (c / (8/P)) mod P for P <= 8 and c mod 8 for P = 16, 32: the eight
// lanes of a quarter-warp then touch eight different 16-byte units mod 128
// bytes, for the copies and for each lane's 128-bit reads of its own pieces.
template <int P>
__device__ __forceinline__ int ring_unit(int c, int q) {
  return P * c + (q ^ (P <= 8 ? ((c / (8 / P)) & (P - 1)) : (c & 7)));
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
// offset that depends on k only through k mod M (M = P/4 for P >= 8, else
// 1), so every copy of a tile is one per-lane base plus a constant.
template <int P>
__device__ __forceinline__ uint32_t ring_piece_off(int lane, int k) {
  constexpr int M = P >= 8 ? P / 4 : 1;
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

// Lane's P pieces of the tile in the slot at byte address slot (aligned to
// 16 P bytes): piece q at (slot + 16 P lane + 16 sw) xor 16 q.
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

// ---------------------------------------------------------- TMA staging
//
// The bf16 G = 128 encode stages its input with the tensor memory
// accelerator: per warp tile one elected lane issues bulk tensor copies of
// 32 rows x 128 bytes (the lanes' slices, two boxes per tile) with the
// 128-byte swizzle, which leaves each lane's 16-byte chunk j of a box row
// at chunk j xor (lane mod 8), so the lanes' 128-bit reads are free of bank
// conflicts; an mbarrier per warp counts the bytes in.  Every wait is
// bounded: on giving up the warp counts the event in g_wait_timeouts
// (fp4_wait_timeouts() reads it) and returns.

__device__ unsigned long long g_wait_timeouts;

constexpr uint32_t kWaitSpins = 1u << 18;  // try_wait rounds before giving up (about 1 s)

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Box {x, y} of the 2-D tensor map into shared memory at dst; its bytes
// complete on mbarrier bar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Lane's P pieces of a TMA-staged tile in the slot at byte address slot
// (1024-byte aligned): piece q is chunk q mod 8 of row `lane` of box q / 8.
template <int P>
__device__ __forceinline__ void tma_read(uint32_t slot, int lane, uint4 v[P]) {
  const uint32_t a = slot + 128u * (uint32_t)lane + 16u * (uint32_t)(lane & 7);
#pragma unroll
  for (int q = 0; q < P; ++q)
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[q].x), "=r"(v[q].y), "=r"(v[q].z), "=r"(v[q].w)
                 : "r"((a + 4096u * (uint32_t)(q >> 3)) ^ (16u * (uint32_t)(q & 7)))
                 : "memory");
}

// ------------------------------------------------------------------ encode
//
// Each lane holds whole chunk pairs of its group: 64 elements (G = 64 and
// 256: L = G/64 lanes per group) or 128 (G = 128: one lane per group).
// Chunk pair m (chunks 2m, 2m + 1) sits in 32 packed pairs
// p[32 h + j] = (chunk 2m element j, chunk 2m + 1 element j), h = m - NP l
// (NP = chunk pairs per lane).  Stages h = 1 .. 16 then pair registers, both
// chunks at once; stage h = 32 pairs the two halves of each register; stage
// h = 64 of G = 128 pairs the lane's two chunk pairs.  For G = 256 the
// stages h = 64, 128 follow a transpose (transpose_wide), after which lane k
// holds positions 8 k .. 8 k + 7 of every chunk pair m as
// p[8 m + b] = (chunk 2m, chunk 2m + 1 at position 8 k + b).
//
// Every product that feeds a packed addition (the squares, the RMS scaling)
// is a packed fma with the runtime -0 addend nz: fma(a, b, -0) = RN(a b)
// exactly, and the compiler cannot fold nz away, so no multiply fuses into
// an add.  More elements per lane mean fewer lanes per group: G = 64 and 128
// need no cross-lane exchange at all.
template <int G>
struct Wide {
  static constexpr int EPL = G == 128 ? 128 : 64;  // elements per lane
  static constexpr int NP = EPL / 64;               // chunk pairs per lane
  static constexpr int L = G / EPL;                 // lanes per group
  static constexpr int B = 32 / L;                  // positions per chunk after the transpose
};

template <int G>
struct WideRow {
  F2 p[16 * Wide<G>::NP * 2];
};

// Transpose tile of the encode (see transpose_wide): C L units per group.
template <int G>
struct WideTile {
  static constexpr int C = 16 * Wide<G>::NP + 1;
  static constexpr int kBytes = Wide<G>::L > 1 ? 16 * C * 32 : 0;  // per warp
};

// Threads per CTA of the encode: 256 (two CTAs per SM at about 120
// registers) for G = 64 and 256; for G = 128, whose lanes hold a whole
// 128-element group, one CTA of 384 threads at up to 170 registers (12
// warps per SM; 256 threads at 238 registers gave 8, and ran 4% slower).
template <int G>
struct EncThreads {
  static constexpr int N = G == 128 ? 384 : 256;
  static constexpr int W = N / 32;
};

// Input pieces per lane and shared memory of the encode: one staging slot
// per warp (bf16: 8 or 16 pieces per lane, fp32 twice that), plus for
// G = 256 the transpose tile.
template <int G, bool kBF16>
struct EncSmem {
  static constexpr int P = Wide<G>::EPL * (kBF16 ? 2 : 4) / 16;
  static constexpr int kSlot = 32 * 16 * P;
  static constexpr int kTile = WideTile<G>::kBytes;
  // slots, transpose tiles, one mbarrier per warp, and room to align the
  // slots to 1024 bytes (the 128-byte swizzle's period)
  static constexpr size_t kSmem = (size_t)EncThreads<G>::W * (kSlot + kTile + 8) + 1024;
};

// TMA staging for the bf16 G = 128 encode (measured faster there; the
// cp.async ring was as fast or faster for the other groups and for fp32).
template <int G, bool kBF16>
constexpr bool enc_tma() {
  return G == 128 && kBF16;
}

// The lane's chunk pairs from its staged pieces: chunk c's 32 elements are
// pieces 4c .. 4c + 3 (bf16) or 8c .. 8c + 7 (fp32).
template <int G, bool kBF16>
__device__ __forceinline__ void unpack_wide(const uint4* v, WideRow<G>& y) {
  constexpr int NP = Wide<G>::NP;
#pragma unroll
  for (int h = 0; h < NP; ++h) {
    if (kBF16) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 a = v[8 * h + q], b = v[8 * h + 4 + q];
        const uint32_t lo[4] = {a.x, a.y, a.z, a.w};
        const uint32_t hi[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = 4 * q + k;  // word i: elements 2i, 2i + 1 of each chunk
          y.p[32 * h + 2 * i] = F2{bf16_lo_(lo[k]), bf16_lo_(hi[k])};
          y.p[32 * h + 2 * i + 1] = F2{bf16_hi_(lo[k]), bf16_hi_(hi[k])};
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 a = v[16 * h + q], b = v[16 * h + 8 + q];
        y.p[32 * h + 4 * q] = F2{__uint_as_float(a.x), __uint_as_float(b.x)};
        y.p[32 * h + 4 * q + 1] = F2{__uint_as_float(a.y), __uint_as_float(b.y)};
        y.p[32 * h + 4 * q + 2] = F2{__uint_as_float(a.z), __uint_as_float(b.z)};
        y.p[32 * h + 4 * q + 3] = F2{__uint_as_float(a.w), __uint_as_float(b.w)};
      }
    }
  }
}

// Transpose of the encode when a group spans L > 1 lanes.  Writer l holds
// chunk pairs NP l + h (h < NP); reader k is to hold positions
// B k .. B k + B - 1 of every chunk pair.  Writer l's unit s for reader k
// (s = h B/2 + u: positions B k + 2u, B k + 2u + 1 of its pair h) goes to
// unit l + L s + C k of the group's region of C L units, C the smallest
// number >= 16 NP that is 1 mod 8; reader k takes it from there into its
// registers for pair NP m + h.  Both sides are a lane base plus a constant,
// and since L s + l covers 0 .. 16 NP - 1 once and C = 1 mod 8, the eight
// lanes of a quarter-warp touch eight different units mod 8 on every access.
template <int G>
__device__ __forceinline__ void transpose_wide(WideRow<G>& y, float4* tile, int lane) {
  constexpr int NP = Wide<G>::NP, L = Wide<G>::L, B = Wide<G>::B, H = B / 2;
  constexpr int C = WideTile<G>::C;
  const int g = lane / L, l = lane % L;
  float4* const st = tile + C * L * g + l;
  const float4* const ld = tile + C * L * g + C * l;
#pragma unroll
  for (int k = 0; k < L; ++k) {
#pragma unroll
    for (int h = 0; h < NP; ++h) {
#pragma unroll
      for (int u = 0; u < H; ++u) {
        const F2 a = y.p[32 * h + B * k + 2 * u], b = y.p[32 * h + B * k + 2 * u + 1];
        st[L * (H * h + u) + C * k] = make_float4(a.x, a.y, b.x, b.y);
      }
    }
  }
  __syncwarp();
#pragma unroll
  for (int m = 0; m < L; ++m) {
#pragma unroll
    for (int h = 0; h < NP; ++h) {
#pragma unroll
      for (int u = 0; u < H; ++u) {
        const float4 v = ld[m + L * (H * h + u)];
        y.p[(NP * m + h) * B + 2 * u] = F2{v.x, v.y};
        y.p[(NP * m + h) * B + 2 * u + 1] = F2{v.z, v.w};
      }
    }
  }
  __syncwarp();
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int m = 1; m < Wide<G>::L; m <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int m = 1; m < Wide<G>::L; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

// The loop walks tiles of 32 lanes' slices, one per warp per grid-stride
// step, warp-uniform so that every lane takes part in the exchanges.  Each
// warp stages its next tile into its one shared slot as soon as it has read
// the current tile out of it (one cp.async group per tile, committed even
// when empty), so the copy runs under the current tile's arithmetic.  Lanes
// past the end compute on zeros and store nothing (the slice count is a
// multiple of L, so a group is entirely inside or entirely past the end).
// Tile indices are 32-bit (the entry point admits fewer than 2^40 elements).
// kTma: the input is staged by TMA through tmap (see above), else by the
// cp.async ring from x.  tx_extra is 0 but for the wait test hook
// (fp4_test_encode_wait_timeout), whose waits never complete.
template <int G, bool kBF16, bool kTma>
__global__ void __launch_bounds__(EncThreads<G>::N, Wide<G>::EPL == 128 ? 1 : 2)
    encode_kernel(const __grid_constant__ CUtensorMap tmap, const void* __restrict__ x,
                  int64_t nslices, uint8_t* __restrict__ packed, float* __restrict__ s1_out,
                  float* __restrict__ s2_out, float nz, uint32_t tx_extra) {
  using W = Wide<G>;
  using M = EncSmem<G, kBF16>;
  constexpr int NP = W::NP, L = W::L, B = W::B, P = M::P, NR = 32 * NP;
  extern __shared__ __align__(1024) uint8_t enc_smem_raw[];
  uint8_t* const enc_smem =
      enc_smem_raw +
      ((1024u - ((uint32_t)__cvta_generic_to_shared(enc_smem_raw) & 1023u)) & 1023u);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t slot =
      (uint32_t)__cvta_generic_to_shared(enc_smem) + (uint32_t)(wid * M::kSlot);
  float4* const tile =
      reinterpret_cast<float4*>(enc_smem + EncThreads<G>::W * M::kSlot + wid * M::kTile);
  const uint32_t bar = (uint32_t)__cvta_generic_to_shared(
      enc_smem + EncThreads<G>::W * (M::kSlot + M::kTile) + 8 * wid);
  constexpr int KB = P / 8;                   // TMA boxes (4 KB) per tile
  constexpr int BX = 128 / (kBF16 ? 2 : 4);   // elements per box row
  const int ntiles = (int)((nslices + 31) >> 5), nfull = (int)(nslices >> 5);
  const int rem = (int)(nslices & 31);
  const int tstride = (int)gridDim.x * EncThreads<G>::W;
  const int64_t step = (int64_t)tstride * M::kSlot;  // input bytes between a warp's tiles
  int t = (int)blockIdx.x * EncThreads<G>::W + wid;
  const uint8_t* src = static_cast<const uint8_t*>(x) + (int64_t)t * M::kSlot;
  if (kTma) {
    if (lane == 0) {
      mbar_init(bar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
  }
  auto stage = [&](int tt, const uint8_t* s) {
    if (kTma) {
      // rows past nslices arrive as zeros
      if (tt < ntiles && lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(bar, KB * 4096 + tx_extra);
#pragma unroll
        for (int b = 0; b < KB; ++b) tma_load_2d(slot + 4096u * b, &tmap, b * BX, 32 * tt, bar);
      }
    } else {
      if (tt < nfull)
        ring_copy_full<P>(slot, s + 16 * lane, lane);
      else if (tt < ntiles)
        ring_copy<P>(slot, s, (nslices - 32 * (int64_t)tt) * (16 * P), lane);
      cp_async_commit();
    }
  };
  const F2 nz2{nz, nz};
  uint32_t phase = 0;
  stage(t, src);
  for (; t < ntiles; t += tstride, src += step) {
    uint4 v[P];
    if (kTma) {
      for (uint32_t spins = 0; !mbar_try_wait(bar, phase);) {
        if (++spins > kWaitSpins) {
          if (lane == 0) atomicAdd(&g_wait_timeouts, 1ull);
          return;
        }
      }
      phase ^= 1u;
      tma_read<P>(slot, lane, v);
    } else {
      cp_async_wait<0>();
      __syncwarp();
      ring_read<P>(slot, lane, v);
    }
    __syncwarp();  // every lane's reads of the slot before its next copy
    stage(t + tstride, src + step);
    WideRow<G> y;
    unpack_wide<G, kBF16>(v, y);
    // RMS: the pairwise tree over adjacent squares, both chunks of a pair side
    // by side (levels 1 - 5), then the pair, the lane's pairs and the lanes
    float pair[NP];
#pragma unroll
    for (int h = 0; h < NP; ++h) {
      F2 sq[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const F2 a = y.p[32 * h + 2 * i], b = y.p[32 * h + 2 * i + 1];
        sq[i] = add2(fma2(a, a, nz2), fma2(b, b, nz2));
      }
#pragma unroll
      for (int w = 16; w > 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w / 2; ++i) sq[i] = add2(sq[2 * i], sq[2 * i + 1]);
      }
      pair[h] = __fadd_rn(sq[0].x, sq[0].y);
    }
    const float ss = group_sum<G>(NP == 2 ? __fadd_rn(pair[0], pair[NP - 1]) : pair[0]);
    const float rms = sqrt_rn(__fmul_rn(ss, 1.0f / (float)G));
    const float inv1 = rms == 0.0f ? 0.0f : rcp_rn(rms);
    const F2 i1 = splat(inv1);
#pragma unroll
    for (int j = 0; j < NR; ++j) y.p[j] = fma2(y.p[j], i1, nz2);
    // stages h = 1 .. 16, h = 32 (the halves), h = 64 inside the lane (G = 128)
#pragma unroll
    for (int hp = 1; hp < 32; hp <<= 1) {
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        if (j & hp) continue;
        const F2 a = y.p[j], b = y.p[j + hp];
        y.p[j] = add2(a, b);
        y.p[j + hp] = sub2(a, b);
      }
    }
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const float a = y.p[j].x, b = y.p[j].y;
      y.p[j] = F2{__fadd_rn(a, b), __fsub_rn(a, b)};
    }
    if (NP == 2) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const F2 a = y.p[j], b = y.p[32 + j];
        y.p[j] = add2(a, b);
        y.p[32 + j] = sub2(a, b);
      }
    }
    if (L > 1) {
      // the stages that pair chunk pairs of different lanes (M, M xor mm)
      transpose_wide<G>(y, tile, lane);
#pragma unroll
      for (int mm = NP; mm < NP * L; mm <<= 1) {
#pragma unroll
        for (int m = 0; m < NP * L; ++m) {
          if (m & mm) continue;
#pragma unroll
          for (int b = 0; b < B; ++b) {
            const F2 a = y.p[m * B + b], c = y.p[(m + mm) * B + b];
            y.p[m * B + b] = add2(a, c);
            y.p[(m + mm) * B + b] = sub2(a, c);
          }
        }
      }
    }
    // normalization and absmax scale into [-6, 6].  z = RN(w c) and
    // max|z| = RN(max|w| c) (RN is monotone).  For G = 64 and 256, c is a
    // power of two: when 2^-20 <= max|z| <= 2^100, RN(z inv2) = RN(w (c inv2))
    // for every element (c inv2 is exact; where w c is normal, z = w c
    // exactly; where it is subnormal, both products are below 2^-100 and
    // round to a zero code of w's sign), so the two scalings fold into one.
    float am = 0.0f;
#pragma unroll
    for (int q = 0; q < NR / 16; ++q) {
      const Row32& h = *reinterpret_cast<const Row32*>(y.p + 16 * q);
      am = fmaxf(am, absmax32(h));
    }
    const float c = wht_norm<G>();
    const float zmax = __fmul_rn(group_max<G>(am), c);
    const float sc2 = div6_rn(zmax);
    const float inv2 = sc2 == 0.0f ? 0.0f : rcp_rn(sc2);
    if (G != 128 && zmax >= 0x1p-20f && zmax <= 0x1p100f) {
      const F2 m = splat(__fmul_rn(inv2, c));
#pragma unroll
      for (int j = 0; j < NR; ++j) y.p[j] = mul2(y.p[j], m);
    } else {
#pragma unroll
      for (int j = 0; j < NR; ++j) y.p[j] = mul2(mul2(y.p[j], splat(c)), splat(inv2));
    }
    if (!(t < nfull || lane < rem)) continue;
    const int l = lane % L;
    const int64_t sl = (int64_t)t * 32 + lane;                    // the lane's slice
    uint8_t* const grp = packed + (int64_t)(W::EPL / 2) * (sl - l);  // the group's codes
    if (L == 1) {
      // the lane's chunks in order, 32 or 64 bytes
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        uint32_t wd[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const F2* q = y.p + 32 * h + 8 * k;
          wd[k] = cvt_e2m1x8(q[0].x, q[1].x, q[2].x, q[3].x, q[4].x, q[5].x, q[6].x, q[7].x);
          wd[4 + k] = cvt_e2m1x8(q[0].y, q[1].y, q[2].y, q[3].y, q[4].y, q[5].y, q[6].y, q[7].y);
        }
        uint4* const o = reinterpret_cast<uint4*>(grp + 32 * h);
        o[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        o[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
      }
    } else {
      // chunk 2M: p[M B + b].x, chunk 2M + 1: .y, positions B l + b: B/2
      // bytes at byte B l / 2 of each chunk's 16-byte row
#pragma unroll
      for (int m = 0; m < NP * L; ++m) {
        const F2* q = y.p + m * B;
        uint32_t wx[B / 8], wy[B / 8];
#pragma unroll
        for (int k = 0; k < B / 8; ++k) {
          wx[k] = cvt_e2m1x8(q[8 * k].x, q[8 * k + 1].x, q[8 * k + 2].x, q[8 * k + 3].x,
                             q[8 * k + 4].x, q[8 * k + 5].x, q[8 * k + 6].x, q[8 * k + 7].x);
          wy[k] = cvt_e2m1x8(q[8 * k].y, q[8 * k + 1].y, q[8 * k + 2].y, q[8 * k + 3].y,
                             q[8 * k + 4].y, q[8 * k + 5].y, q[8 * k + 6].y, q[8 * k + 7].y);
        }
        uint8_t* const r0 = grp + 32 * m + (B / 2) * l;
        if (B == 16) {
          *reinterpret_cast<uint2*>(r0) = make_uint2(wx[0], wx[1]);
          *reinterpret_cast<uint2*>(r0 + 16) = make_uint2(wy[0], wy[1]);
        } else {
          *reinterpret_cast<uint32_t*>(r0) = wx[0];
          *reinterpret_cast<uint32_t*>(r0 + 16) = wy[0];
        }
      }
    }
    if (l == 0) {
      const int64_t gi = sl / L;
      s1_out[gi] = rms;
      s2_out[gi] = sc2;
    }
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
  static constexpr size_t kSmem = (size_t)kWarps * (NS * kSlot + TTile::kBytes);
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
// encode kernels; tile indices are 32-bit likewise.  The bf16-output kernel
// for G = 256 is held to 64 registers (four CTAs per SM); for G = 64 and 128
// three CTAs at 71-72 registers measured faster.
template <int G, bool kBF16Out>
__global__ void __launch_bounds__(kThreads, (kBF16Out && G == 256) ? 4 : 1)
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
      reinterpret_cast<float4*>(dec_smem + kWarps * NS * R::kSlot + wid * TTile::kBytes);
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (looked up once), or null.
EncodeTiledFn encode_tiled_fn() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// The encode's input as a 2-D tensor for TMA: nslices rows of P 16-byte
// pieces, read in boxes of 32 rows x 128 bytes with the 128-byte swizzle.
template <bool kBF16, int P>
bool encode_tensor_map(CUtensorMap* m, const void* x, int64_t nslices) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  constexpr int esize = kBF16 ? 2 : 4;
  const cuuint64_t gdim[2] = {(cuuint64_t)P * 16 / esize, (cuuint64_t)nslices};
  const cuuint64_t gstride[1] = {(cuuint64_t)P * 16};
  const cuuint32_t box[2] = {128 / esize, 32};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
             const_cast<void*>(x), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G, bool kBF16>
fp4_status launch_encode_t(const void* x, int64_t nchunks, uint8_t* packed, float* s1, float* s2,
                           cudaStream_t s, uint32_t tx_extra = 0) {
  constexpr size_t smem = EncSmem<G, kBF16>::kSmem;
  static_assert(smem <= 227 * 1024, "one CTA's shared memory must fit an SM");
  const int64_t nslices = nchunks / (Wide<G>::EPL / kE);
  alignas(64) CUtensorMap m = {};
  if constexpr (enc_tma<G, kBF16>()) {
    // TMA row coordinates are 32-bit: past 2^31 slices the cp.async ring stages
    if (nslices < ((int64_t)1 << 31)) {
      if (!allow_dynamic_smem<encode_kernel<G, kBF16, true>>(smem)) return FP4_ERR_CUDA;
      if (!encode_tensor_map<kBF16, EncSmem<G, kBF16>::P>(&m, x, nslices)) return FP4_ERR_CUDA;
      return launch<encode_kernel<G, kBF16, true>>(nslices, EncThreads<G>::N, smem, s, m, x,
                                                   nslices, packed, s1, s2, -0.0f, tx_extra);
    }
  }
  if (!allow_dynamic_smem<encode_kernel<G, kBF16, false>>(smem)) return FP4_ERR_CUDA;
  if (tx_extra != 0) return FP4_ERR_ARG;  // only the TMA path has the waits
  return launch<encode_kernel<G, kBF16, false>>(nslices, EncThreads<G>::N, smem, s, m, x,
                                                nslices, packed, s1, s2, -0.0f, 0u);
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
  static_assert(smem <= 227 * 1024, "one CTA's shared memory must fit an SM");
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

fp4_status fp4_test_encode_wait_timeout(const void* x, int64_t rows, int64_t cols,
                                        uint8_t* packed, float* s1, float* s2, void* stream) {
  if (rows <= 0 || cols <= 0 || cols % 128 != 0 || rows > ((int64_t)1 << 24) / cols)
    return FP4_ERR_SHAPE;
  if (!x || !packed || !s1 || !s2) return FP4_ERR_NULL;
  if (!aligned(x, 32) || !aligned(packed, 16) || !aligned(s1, 4) || !aligned(s2, 4))
    return FP4_ERR_ALIGN;
  return launch_encode_t<128, true>(x, rows * cols / kE, packed, s1, s2, as_stream(stream), 16u);
}

uint64_t fp4_wait_timeouts(void) {
  unsigned long long v = 0;
  if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) return UINT64_MAX;
  return (uint64_t)v;
}

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
