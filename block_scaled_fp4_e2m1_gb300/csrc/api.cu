// api.cu -- status strings, version, launch count and the host-side segment
// offset helper of the C ABI.
#include <cuda_runtime.h>

#include <atomic>

#include "host_common.h"

namespace fp4 {

std::atomic<uint64_t> g_kernel_launches{0};

int sm_count() {
  // Device properties do not change; cache them for up to 64 devices.
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 1;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace fp4

extern "C" {

const char* fp4_status_string(int status) {
  switch (status) {
    case FP4_OK: return "ok";
    case FP4_ERR_NULL: return "a required pointer is NULL";
    case FP4_ERR_ALIGN: return "a pointer is not aligned as required";
    case FP4_ERR_SHAPE: return "a size is negative or breaks its divisibility rule";
    case FP4_ERR_DTYPE: return "unknown dtype";
    case FP4_ERR_ARG: return "an argument is out of range";
    case FP4_ERR_CUDA: return "a CUDA launch failed";
    case FP4_ERR_INTERNAL: return "internal error";
    default: return "unknown status";
  }
}

int fp4_abi_version(void) { return FP4CODEC_ABI_VERSION; }

uint64_t fp4_kernel_launches(void) {
  return fp4::g_kernel_launches.load(std::memory_order_relaxed);
}

fp4_status fp4_seg_scale_offsets(const int64_t* host_row_off, int32_t num_segments,
                                 int64_t* host_scale_off) {
  if (!host_row_off || !host_scale_off) return FP4_ERR_NULL;
  if (num_segments < 0) return FP4_ERR_SHAPE;
  int64_t acc = 0;
  host_scale_off[0] = 0;
  for (int32_t e = 0; e < num_segments; ++e) {
    int64_t n = host_row_off[e + 1] - host_row_off[e];
    if (n < 0) return FP4_ERR_SHAPE;
    acc += (n + 127) / 128;
    host_scale_off[e + 1] = acc;
  }
  return FP4_OK;
}

}  // extern "C"
