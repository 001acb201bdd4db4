// Device side of the synthetic-input generator: the same counter-based
// generator as the host side (philox_ih.h), writing straight into device
// memory so that multi-gigabyte synthetic models are made in milliseconds.
// Holds no arithmetic of the decode method.
#include <cuda_runtime.h>
#include <stdint.h>
#include "philox_ih.h"

namespace {

__global__ void fill_normal_kernel(float* __restrict__ out, uint64_t n, uint64_t first,
                                   uint32_t seed, uint32_t stream, float scale, float mean) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = tqs_normal_at(seed, stream, first + i, scale);
    out[i] = (mean != 0.0f) ? __fadd_rn(mean, v) : v;
  }
}

__global__ void fill_uniform_kernel(int32_t* __restrict__ out, uint64_t n, uint64_t first,
                                    uint32_t seed, uint32_t stream, uint32_t bound) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = (int32_t)tqs_uniform_below(seed, stream, first + i, bound);
}

unsigned grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 32ull) g = 152ull * 32ull;
  if (g == 0) g = 1;
  return (unsigned)g;
}

}  // namespace

extern "C" int tqs_dev_fill_normal(float* out, uint64_t n, uint64_t first, uint32_t seed,
                                   uint32_t stream, float scale, float mean, void* cuda_stream) {
  if (n == 0) return 0;
  if (out == nullptr) return 1;
  fill_normal_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(out, n, first, seed,
                                                                          stream, scale, mean);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

extern "C" int tqs_dev_fill_uniform_below(int32_t* out, uint64_t n, uint64_t first,
                                          uint32_t seed, uint32_t stream, uint32_t bound,
                                          void* cuda_stream) {
  if (n == 0) return 0;
  if (out == nullptr || bound == 0) return 1;
  fill_uniform_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(out, n, first, seed,
                                                                           stream, bound);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
