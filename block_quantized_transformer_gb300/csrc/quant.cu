// Block formats on the GPU: encode f32 -> GGUF-order Q8_0/Q4_0 blocks or
// MLX-layout affine 4-bit groups, repack either into the tiled layout the
// GEMV streams (see kernels.cuh), decode rows of it to f32, and gather
// embedding rows.
//
// The formats are the workload descriptions' Q8_0 (fp16 d = max|w|/127,
// int8 q = round(w/d), value d*q) and Q4_0 (fp16 d = m/-8 at the signed
// extreme, q = clamp(round(w/d)+8, 0, 15), value d*(q-8)).  Encoding decisions
// are taken in f32 exactly as the header tq.h states; decoding is exact.
// Affine 4-bit ("Alchemize PyTensor ... Gemma 3n": W = q s + b per group of
// inputs, eight 4-bit values per uint32 word, bf16 scale and bias): groups of
// 64, s = (max - min) / 15, b = min, q = round((w - b) / s) decided in f32,
// s and b stored as bf16; decoding q s + b rounds once in f32.
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace tq {

// ----------------------------------------------------------------- encode --

__device__ __forceinline__ float round_half_away(float v) {
  float t = truncf(v);
  if (fabsf(v - t) >= 0.5f) t += copysignf(1.0f, v);
  return t;
}

// One warp per block of 32 weights; lane j holds weight j.
template <int WT>
__global__ void quantize_kernel(const float* __restrict__ w, int64_t n_blocks,
                                uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (; blk < n_blocks; blk += stride) {
    const float x = w[blk * 32 + lane];
    float d;
    if (WT == TQ_Q8_0) {
      const float amax = warp_max(fabsf(x));
      d = amax / 127.0f;
    } else {
      // first element of largest magnitude: larger |x| wins, then lower index
      unsigned long long key =
          ((unsigned long long)__float_as_uint(fabsf(x)) << 32) | (unsigned)(31 - lane);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
        key = other > key ? other : key;
      }
      const int src = 31 - (int)(key & 0xffffffffull);
      const float m = __shfl_sync(0xffffffffu, x, src);
      d = m / -8.0f;
    }
    int q;
    if (WT == TQ_Q8_0) {
      q = d == 0.0f ? 0 : (int)round_half_away(x / d);
      q = max(-127, min(127, q));
    } else {
      q = d == 0.0f ? 8 : (int)round_half_away(x / d) + 8;
      q = max(0, min(15, q));
    }
    constexpr int BB = WT == TQ_Q8_0 ? 34 : 18;
    uint8_t* o = out + blk * BB;
    if (lane == 0) {
      // blocks start at even offsets (34 and 18 are even): one 16-bit store
      *reinterpret_cast<uint16_t*>(o) = __half_as_ushort(__float2half_rn(d));
    }
    if (WT == TQ_Q8_0) {
      o[2 + lane] = (uint8_t)(int8_t)q;
    } else {
      const int hi = __shfl_down_sync(0xffffffffu, q, 16);
      if (lane < 16) o[2 + lane] = (uint8_t)(q | (hi << 4));
    }
  }
}

// One warp per group of 64 inputs: lane l holds inputs l and l + 32.
__global__ void quantize_affine4_kernel(const float* __restrict__ w, int64_t n_groups, uint32_t* __restrict__ words,
                                        uint16_t* __restrict__ scales, uint16_t* __restrict__ biases) {
  const int lane = threadIdx.x & 31;
  int64_t grp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (; grp < n_groups; grp += stride) {
    const float x0 = w[grp * 64 + lane], x1 = w[grp * 64 + 32 + lane];
    float lo = fminf(x0, x1), hi = fmaxf(x0, x1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const float s = (hi - lo) / 15.0f;
    const float b = lo;
    int q0 = 0, q1 = 0;
    if (s != 0.0f) {
      q0 = max(0, min(15, (int)round_half_away((x0 - b) / s)));
      q1 = max(0, min(15, (int)round_half_away((x1 - b) / s)));
    }
    // element 8w + i of the group in bits 4i of word w: lanes 8w .. 8w+7 (w < 4)
    // hold the first half's words, the same lanes' second values words 4 .. 7
    uint32_t p0 = (uint32_t)q0 << (4 * (lane & 7)), p1 = (uint32_t)q1 << (4 * (lane & 7));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      p0 |= __shfl_xor_sync(0xffffffffu, p0, o);
      p1 |= __shfl_xor_sync(0xffffffffu, p1, o);
    }
    if ((lane & 7) == 0) {
      words[grp * 8 + (lane >> 3)] = p0;
      words[grp * 8 + 4 + (lane >> 3)] = p1;
    }
    if (lane == 0) {
      scales[grp] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
      biases[grp] = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    }
  }
}

// ----------------------------------------------------------------- repack --

// One thread per (row, block) of the padded matrix.  GGUF blocks start at even
// offsets (34 and 18 are even), so they are read as 16-bit words; rows past
// the end of the matrix (tile padding) get zero codes and zero scales.
template <int WT>
__global__ void repack_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t nb,
                              uint8_t* __restrict__ qs, uint16_t* __restrict__ d) {
  const int64_t n = tiled_rows(rows) * nb;
  constexpr int NW = WT == TQ_Q8_0 ? 8 : 4;   // 32-bit words of codes per block
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb, blk = i % nb;
    uint32_t v[NW];
    uint16_t dv = 0;
    if (r < rows) {
      const uint16_t* b = src + i * (1 + 2 * NW);
      dv = b[0];
#pragma unroll
      for (int k = 0; k < NW; ++k) v[k] = (uint32_t)b[1 + 2 * k] | ((uint32_t)b[2 + 2 * k] << 16);
    } else {
#pragma unroll
      for (int k = 0; k < NW; ++k) v[k] = 0u;
    }
    d[tiled_d_index(r, blk, nb)] = dv;
#pragma unroll
    for (int k = 0; k < NW; ++k)
      *reinterpret_cast<uint32_t*>(qs + tiled_qs_offset(WT, r, blk, nb, k)) = v[k];
  }
}

// One thread per (row, 32-input block) of the padded matrix: the block's 32
// codes from the MLX words rearranged as a Q4_0 block's bytes (q[j] |
// q[j+16] << 4), and the group's scale (even block) or bias (odd block).
__global__ void repack_affine4_kernel(const uint32_t* __restrict__ words, const uint16_t* __restrict__ scales,
                                      const uint16_t* __restrict__ biases, int64_t rows, int64_t nb,
                                      uint8_t* __restrict__ qs, uint16_t* __restrict__ d) {
  const int64_t n = tiled_rows(rows) * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb, blk = i % nb;
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    uint16_t dv = 0;
    if (r < rows) {
      const uint32_t* wr = words + r * (nb * 4) + blk * 4;  // inputs 32 blk .. 32 blk + 31
      uint32_t q[32];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t x = wr[w];
#pragma unroll
        for (int k = 0; k < 8; ++k) q[8 * w + k] = (x >> (4 * k)) & 15u;
      }
#pragma unroll
      for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int k = 0; k < 4; ++k) v[w] |= (q[4 * w + k] | (q[4 * w + k + 16] << 4)) << (8 * k);
      const int64_t grp = r * (nb / 2) + blk / 2;
      dv = (blk & 1) ? biases[grp] : scales[grp];
    }
    d[tiled_d_index(r, blk, nb)] = dv;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint32_t*>(qs + tiled_qs_offset(TQ_AFFINE4, r, blk, nb, k)) = v[k];
  }
}

// --------------------------------------------------------------- decoding --

// Decode block `blk` of row `row` into 32 f32 values: d * code (exact), or
// for AFFINE4 q * s + b with one rounding.
template <int WT>
__device__ __forceinline__ void decode_block(const uint8_t* qs, const uint16_t* dptr, int64_t row,
                                             int64_t nb, int64_t blk, float* out32) {
  const float d = half_bits_to_float(dptr[tiled_d_index(row, blk, nb)]);
  if (WT == TQ_AFFINE4) {
    const float s = bf16_bits_to_float(dptr[tiled_d_index(row, blk & ~1ll, nb)]);
    const float b = bf16_bits_to_float(dptr[tiled_d_index(row, blk | 1ll, nb)]);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t word = *reinterpret_cast<const uint32_t*>(qs + tiled_qs_offset(WT, row, blk, nb, w));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t byte = (word >> (8 * k)) & 0xffu;
        out32[4 * w + k] = fmaf((float)(byte & 0xf), s, b);
        out32[4 * w + k + 16] = fmaf((float)(byte >> 4), s, b);
      }
    }
  } else if (WT == TQ_Q4_0) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t word = *reinterpret_cast<const uint32_t*>(qs + tiled_qs_offset(WT, row, blk, nb, w));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t byte = (word >> (8 * k)) & 0xffu;
        out32[4 * w + k] = d * (float)((int)(byte & 0xf) - 8);
        out32[4 * w + k + 16] = d * (float)((int)(byte >> 4) - 8);
      }
    }
  } else {
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint32_t word = *reinterpret_cast<const uint32_t*>(qs + tiled_qs_offset(WT, row, blk, nb, w));
#pragma unroll
      for (int k = 0; k < 4; ++k) out32[4 * w + k] = d * (float)(int8_t)((word >> (8 * k)) & 0xffu);
    }
  }
}

template <int WT>
__global__ void dequant_kernel(const uint8_t* __restrict__ qs, const uint16_t* __restrict__ d,
                               int64_t nb, int64_t row0, int64_t n_rows, float* __restrict__ out) {
  const int64_t n = n_rows * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb, c = i % nb;
    float v[32];
    decode_block<WT>(qs, d, row0 + r, nb, c, v);
    float4* o = reinterpret_cast<float4*>(out + (r * nb + c) * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
}

// x[t][:] = decoded row tokens[t] of the embedding; ids out of range give
// zeros and set TQ_DEV_BAD_TOKEN.  One CTA per token.
template <int WT>
__global__ void embed_kernel(const uint8_t* __restrict__ qs, const uint16_t* __restrict__ d,
                             int vocab, int hidden, const int32_t* __restrict__ tokens,
                             float* __restrict__ x, uint32_t* status,
                             unsigned long long* argmax_keys, int n_keys) {
  grid_dep_launch();
  grid_dep_wait();  // x and the argmax keys may still be read by the preceding kernel
  const int t = blockIdx.x;
  const int nb = hidden / 32;
  const int tok = tokens[t];
  const bool ok = tok >= 0 && tok < vocab;
  if (!ok && threadIdx.x == 0) set_status(status, TQ_DEV_BAD_TOKEN);
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    float v[32];
    if (ok) {
      decode_block<WT>(qs, d, tok, nb, c, v);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = 0.0f;
    }
    float4* o = reinterpret_cast<float4*>(x + (int64_t)t * hidden + c * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
  // the head's argmax keys are reset here, at the start of every step
  if (argmax_keys != nullptr && t == 0)
    for (int i = threadIdx.x; i < n_keys; i += blockDim.x) argmax_keys[i] = 0ull;
}

static unsigned grid_1d(int64_t n, int per_cta) {
  int64_t g = (n + per_cta - 1) / per_cta;
  if (g > (int64_t)kNumSMs * 64) g = (int64_t)kNumSMs * 64;
  return (unsigned)(g < 1 ? 1 : g);
}

cudaError_t launch_quantize(int wtype, const float* w, int64_t n_blocks, void* out, cudaStream_t s) {
  const unsigned g = grid_1d(n_blocks * 32, 256);
  if (wtype == TQ_Q8_0)
    quantize_kernel<TQ_Q8_0><<<g, 256, 0, s>>>(w, n_blocks, (uint8_t*)out);
  else
    quantize_kernel<TQ_Q4_0><<<g, 256, 0, s>>>(w, n_blocks, (uint8_t*)out);
  return cudaGetLastError();
}

cudaError_t launch_repack(int wtype, const void* src, int64_t rows, int64_t nb, void* qs,
                          uint16_t* d, cudaStream_t s) {
  const unsigned g = grid_1d(tiled_rows(rows) * nb, 256);
  if (wtype == TQ_Q8_0)
    repack_kernel<TQ_Q8_0><<<g, 256, 0, s>>>((const uint16_t*)src, rows, nb, (uint8_t*)qs, d);
  else
    repack_kernel<TQ_Q4_0><<<g, 256, 0, s>>>((const uint16_t*)src, rows, nb, (uint8_t*)qs, d);
  return cudaGetLastError();
}

cudaError_t launch_quantize_affine4(const float* w, int64_t rows, int64_t cols, uint32_t* words, uint16_t* scales,
                                    uint16_t* biases, cudaStream_t s) {
  const int64_t n_groups = rows * (cols / 64);
  quantize_affine4_kernel<<<grid_1d(n_groups * 32, 256), 256, 0, s>>>(w, n_groups, words, scales, biases);
  return cudaGetLastError();
}

cudaError_t launch_repack_affine4(const uint32_t* words, const uint16_t* scales, const uint16_t* biases,
                                  int64_t rows, int64_t cols, void* qs, uint16_t* d, cudaStream_t s) {
  const int64_t nb = cols / 32;
  repack_affine4_kernel<<<grid_1d(tiled_rows(rows) * nb, 256), 256, 0, s>>>(words, scales, biases, rows, nb,
                                                                            (uint8_t*)qs, d);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int wtype, const void* qs, const uint16_t* d, int64_t nb, int64_t row0,
                           int64_t n_rows, float* out, cudaStream_t s) {
  const unsigned g = grid_1d(n_rows * nb, 256);
  if (wtype == TQ_Q8_0)
    dequant_kernel<TQ_Q8_0><<<g, 256, 0, s>>>((const uint8_t*)qs, d, nb, row0, n_rows, out);
  else if (wtype == TQ_AFFINE4)
    dequant_kernel<TQ_AFFINE4><<<g, 256, 0, s>>>((const uint8_t*)qs, d, nb, row0, n_rows, out);
  else
    dequant_kernel<TQ_Q4_0><<<g, 256, 0, s>>>((const uint8_t*)qs, d, nb, row0, n_rows, out);
  return cudaGetLastError();
}

cudaError_t launch_embed(int wtype, const void* qs, const uint16_t* d, int vocab, int hidden,
                         const int32_t* tokens, int n_tokens, float* x, uint32_t* status,
                         unsigned long long* argmax_keys, int n_keys, cudaStream_t s) {
  const int threads = hidden / 32 < 128 ? 32 * ((hidden / 32 + 31) / 32) : 128;
  if (wtype == TQ_Q8_0)
    return launch_k(embed_kernel<TQ_Q8_0>, dim3(n_tokens), dim3(threads), 0, s, (const uint8_t*)qs, d,
                    vocab, hidden, tokens, x, status, argmax_keys, n_keys);
  if (wtype == TQ_AFFINE4)
    return launch_k(embed_kernel<TQ_AFFINE4>, dim3(n_tokens), dim3(threads), 0, s, (const uint8_t*)qs, d,
                    vocab, hidden, tokens, x, status, argmax_keys, n_keys);
  return launch_k(embed_kernel<TQ_Q4_0>, dim3(n_tokens), dim3(threads), 0, s, (const uint8_t*)qs, d,
                  vocab, hidden, tokens, x, status, argmax_keys, n_keys);
}

}  // namespace tq
