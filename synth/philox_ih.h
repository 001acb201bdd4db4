/* Seeded synthetic-input generator shared by the oracle side and the GPU side.
 *
 * This header holds no arithmetic of the decode method: it only turns
 * (seed, stream, element index) into numbers, so that any element of any
 * synthetic tensor can be produced independently, on the host or on the GPU,
 * bit for bit identically.
 *
 *  - Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and
 *    Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): a 128-bit
 *    counter and a 64-bit key, ten rounds of two 32x32->64 multiplies, key
 *    bumped by the Weyl constants between rounds.
 *  - Approximately normal values: the Irwin-Hall sum of the eight 16-bit
 *    halves of one Philox output, centred and scaled to unit variance.  The
 *    sum is an exact integer; the only floating-point step is one
 *    round-to-nearest f32 multiply by a constant rounded once from double, so
 *    every machine and the GPU produce the same f32 bits.
 *  - Uniform integers in [0, n): the high 32 bits of word0 * n.
 *
 * Compiled as plain C by gcc (host library) and as CUDA by nvcc (device
 * kernels); nothing here depends on the compiler.
 */
#ifndef TQ_SYNTH_PHILOX_IH_H
#define TQ_SYNTH_PHILOX_IH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define TQS_FN static __host__ __device__ __forceinline__
#else
#define TQS_FN static inline
#endif

#define TQS_PHILOX_M0 0xD2511F53u
#define TQS_PHILOX_M1 0xCD9E8D57u
#define TQS_PHILOX_W0 0x9E3779B9u
#define TQS_PHILOX_W1 0xBB67AE85u

/* Sum of eight discrete uniforms on {0..65535}: mean 8 * 65535 / 2. */
#define TQS_IH8_MEAN 262140

TQS_FN void tqs_philox4x32_10(const uint32_t ctr[4], uint32_t k0, uint32_t k1,
                              uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += TQS_PHILOX_W0;
      k1 += TQS_PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)TQS_PHILOX_M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)TQS_PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* The four Philox words for element `idx` of stream `stream` under `seed`. */
TQS_FN void tqs_words(uint32_t seed, uint32_t stream, uint64_t idx, uint32_t w[4]) {
  uint32_t ctr[4];
  ctr[0] = (uint32_t)idx;
  ctr[1] = (uint32_t)(idx >> 32);
  ctr[2] = 0u;
  ctr[3] = 0u;
  tqs_philox4x32_10(ctr, seed, stream, w);
}

/* Centred Irwin-Hall(8) integer, in [-262140, 262140]. */
TQS_FN int32_t tqs_ih8_centred(const uint32_t w[4]) {
  int32_t s = 0;
  for (int i = 0; i < 4; ++i) s += (int32_t)(w[i] & 0xFFFFu) + (int32_t)(w[i] >> 16);
  return s - TQS_IH8_MEAN;
}

/* Element `idx` of a N(0, sigma)-like stream: (float)centred * scale, where
 * scale = (float)(sigma / sd(IH8)) is precomputed by the caller with
 * tqs_normal_scale().  One f32 multiply, round to nearest even. */
TQS_FN float tqs_normal_at(uint32_t seed, uint32_t stream, uint64_t idx, float scale) {
  uint32_t w[4];
  tqs_words(seed, stream, idx, w);
  return (float)tqs_ih8_centred(w) * scale;
}

/* Uniform integer in [0, n) for element `idx`. */
TQS_FN uint32_t tqs_uniform_below(uint32_t seed, uint32_t stream, uint64_t idx, uint32_t n) {
  uint32_t w[4];
  tqs_words(seed, stream, idx, w);
  return (uint32_t)(((uint64_t)w[0] * (uint64_t)n) >> 32);
}

#endif /* TQ_SYNTH_PHILOX_IH_H */
