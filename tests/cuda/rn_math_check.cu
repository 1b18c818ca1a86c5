// rn_math_check.cu -- compares the fast correctly rounded routines of
// rn_math.cuh with the CUDA intrinsics on every fp32 bit pattern of a
// range.  Usage: rn_math_check <lo> <hi> (hex bit patterns, hi exclusive);
// prints one line "rcp <n> div6 <n> sqrt <n>" of mismatch counts.
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include <cuda_runtime.h>

#include "rn_math.cuh"

__global__ void check(uint32_t lo, uint32_t n, unsigned long long* bad) {
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float x = __uint_as_float(lo + i);
    if (__float_as_uint(fp4::rcp_rn(x)) != __float_as_uint(__frcp_rn(x))) atomicAdd(&bad[0], 1ull);
    if (__float_as_uint(fp4::div6_rn(x)) != __float_as_uint(__fdiv_rn(x, 6.0f)))
      atomicAdd(&bad[1], 1ull);
    if (__float_as_uint(fp4::sqrt_rn(x)) != __float_as_uint(__fsqrt_rn(x))) atomicAdd(&bad[2], 1ull);
  }
}

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  const uint32_t lo = (uint32_t)strtoul(argv[1], nullptr, 16);
  const uint32_t hi = (uint32_t)strtoul(argv[2], nullptr, 16);
  if (hi <= lo) return 2;
  unsigned long long* bad = nullptr;
  if (cudaMalloc(&bad, 3 * sizeof(unsigned long long)) != cudaSuccess) return 1;
  cudaMemset(bad, 0, 3 * sizeof(unsigned long long));
  check<<<152 * 8, 256>>>(lo, hi - lo, bad);
  unsigned long long h[3] = {0, 0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  cudaMemcpy(h, bad, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(bad);
  printf("rcp %llu div6 %llu sqrt %llu\n", h[0], h[1], h[2]);
  return 0;
}
