// host_common.h -- argument checks and launch bookkeeping shared by the
// C-ABI entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/fp4codec.h"

namespace fp4 {

// Process-wide count of kernels launched by this library.
extern std::atomic<uint64_t> g_kernel_launches;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Number of SMs of the current device (cached per device).
int sm_count();

// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory (at least 1).
template <typename K>
inline int occupancy(K kernel, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
      n < 1)
    n = 1;
  return n;
}

// Opt `Kernel` in to `smem` bytes of dynamic shared memory (once per
// process; needed above 48 KB).
template <auto Kernel>
inline bool allow_dynamic_smem(size_t smem) {
  static const bool ok =
      smem <= 48 * 1024 ||
      cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
          cudaSuccess;
  return ok;
}

// CTAs of `Kernel` resident on the whole GPU at once (one full wave).
template <auto Kernel>
inline int64_t wave_ctas(int threads, size_t smem) {
  static const int occ = occupancy(Kernel, threads, smem);
  return (int64_t)sm_count() * occ;
}

// Grid for a grid-stride loop over `units` thread-level work units: one
// thread per unit up to one full wave of resident CTAs on every SM.
template <auto Kernel>
inline unsigned grid_for_kernel(int64_t units, int threads, size_t smem) {
  int64_t want = (units + threads - 1) / threads;
  const int64_t cap = wave_ctas<Kernel>(threads, smem);
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (unsigned)want;
}

// Status of the launch just enqueued (counts it when it succeeded).
inline fp4_status after_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return FP4_ERR_CUDA;
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return FP4_OK;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool dtype_ok(int d) { return d == FP4_F32 || d == FP4_BF16; }
inline int64_t dtype_size(int d) { return d == FP4_F32 ? 4 : 2; }

// Launch `Kernel` over `units` thread-level units (grid-stride) on stream s.
template <auto Kernel, typename... Args>
inline fp4_status launch(int64_t units, int threads, size_t smem, cudaStream_t s, Args... args) {
  const unsigned grid = grid_for_kernel<Kernel>(units, threads, smem);
  Kernel<<<grid, threads, smem, s>>>(args...);
  return after_launch();
}

}  // namespace fp4
