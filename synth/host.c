/* Host side of the synthetic-input generator: fills host arrays from the
 * counter-based generator in philox_ih.h, in parallel over elements.  Used by
 * the oracle's tests and by the benchmark's CPU baseline; holds no arithmetic
 * of the decode method. */
#include <stdint.h>
#include <stddef.h>
#include "philox_ih.h"

void tqs_host_fill_normal(float* out, uint64_t n, uint64_t first, uint32_t seed,
                          uint32_t stream, float scale, float mean) {
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < nn; ++i) {
    float v = tqs_normal_at(seed, stream, first + (uint64_t)i, scale);
    out[i] = (mean != 0.0f) ? mean + v : v;
  }
}

void tqs_host_fill_uniform_below(int32_t* out, uint64_t n, uint64_t first, uint32_t seed,
                                 uint32_t stream, uint32_t bound) {
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < nn; ++i)
    out[i] = (int32_t)tqs_uniform_below(seed, stream, first + (uint64_t)i, bound);
}

void tqs_host_philox(const uint32_t ctr[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
  tqs_philox4x32_10(ctr, k0, k1, out);
}
