// Temperature / top-p sampling on the device ("Всередині LLM: чисте виконання
// на Python для Qwen3-0.6B на MLX", step 8, sample(logits, temperature,
// top_p)): temperature 0 is the argmax (lowest index on ties); otherwise the
// tempered softmax's tokens in descending order of probability (ties by
// ascending index), the smallest prefix whose cumulative probability reaches
// top_p kept and renormalised, and the draw is the first kept token whose
// cumulative probability exceeds u (a uniform number the caller supplies).
//
// One CTA per row, no sort: both decisions are weighted quantiles of the
// order, found by a radix select over the 32-bit order-preserving key of the
// logit (four passes of 8 bits, each a histogram of the unnormalised mass
// exp2((l - max) log2(e) / T) of the tokens that share the key's leading
// bits, summed in f64), then, among tokens of exactly equal logit, a
// count-based select over the index bits.  The row is read from L2 once per
// pass.
#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace tq {
namespace smp {

constexpr int kThreads = 1024;

struct Hist {
  double mass[256];  // f64 sums: over 151936 tokens f32 sums would move a draw by tens of tokens
  unsigned cnt[256];
};

__device__ __forceinline__ float block_max(float v, float* sh) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float x = sh[threadIdx.x];
    x = warp_max(x);
    if (threadIdx.x == 0) sh[32] = x;
  }
  __syncthreads();
  const float r = sh[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ double block_sum(double v, double* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    double x = sh[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (threadIdx.x == 0) sh[32] = x;
  }
  __syncthreads();
  const double r = sh[32];
  __syncthreads();
  return r;
}

// Result of a weighted quantile: the key of the token where the cumulative
// mass (descending order) reaches the target, the mass of all tokens with a
// larger key, and the number and mass of the tokens that share the key.
struct Quantile {
  uint32_t key;
  double above;
  unsigned n_tie;
  double m_tie;
};

// First token (descending key order) whose inclusive cumulative mass reaches
// `target` (>= when !strict, > when strict); if rounding leaves the total
// below the target, the last token.
__device__ Quantile select_value(const float* row, int V, float lmax, float sc, double target, bool strict,
                                 Hist* h) {
  __shared__ uint32_t s_prefix;
  __shared__ double s_above;
  __shared__ unsigned s_n;
  __shared__ double s_m;
  if (threadIdx.x == 0) {
    s_prefix = 0u;
    s_above = 0.f;
  }
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += kThreads) {
      h->mass[b] = 0.0;
      h->cnt[b] = 0u;
    }
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int i = threadIdx.x; i < V; i += kThreads) {
      const float l = row[i];
      const uint32_t key = float_order_key(l);
      if (shift < 24 && (key >> (shift + 8)) != (prefix >> (shift + 8))) continue;
      const int b = (int)((key >> shift) & 255u);
      atomicAdd(&h->mass[b], (double)exp2f((l - lmax) * sc));
      atomicAdd(&h->cnt[b], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      double cum = s_above;
      int chosen = -1, lowest = -1;
      double cum_low = cum;
      for (int b = 255; b >= 0; --b) {
        if (h->cnt[b] == 0u) continue;
        const double nc = cum + h->mass[b];
        if (strict ? nc > target : nc >= target) {
          chosen = b;
          break;
        }
        lowest = b;
        cum_low = cum;
        cum = nc;
      }
      if (chosen < 0) {  // the total stays below the target: the last token
        chosen = lowest;
        cum = cum_low;
      }
      s_above = cum;
      s_prefix = prefix | ((uint32_t)chosen << shift);
      s_n = h->cnt[chosen];
      s_m = h->mass[chosen];
    }
    __syncthreads();
  }
  Quantile q;
  q.key = s_prefix;
  q.above = s_above;
  q.n_tie = s_n;
  q.m_tie = s_m;
  __syncthreads();
  return q;
}

// The r-th (1-based) lowest index among the tokens whose key equals `key`.
__device__ int select_tie_index(const float* row, int V, uint32_t key, unsigned r, Hist* h) {
  __shared__ uint32_t s_prefix;
  __shared__ unsigned s_before;
  if (threadIdx.x == 0) {
    s_prefix = 0u;
    s_before = 0u;
  }
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += kThreads) h->cnt[b] = 0u;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int i = threadIdx.x; i < V; i += kThreads) {
      if (float_order_key(row[i]) != key) continue;
      const uint32_t ui = (uint32_t)i;
      if (shift < 24 && (ui >> (shift + 8)) != (prefix >> (shift + 8))) continue;
      atomicAdd(&h->cnt[(ui >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned before = s_before;
      int chosen = 255;
      for (int b = 0; b < 256; ++b) {  // ascending index
        if (before + h->cnt[b] >= r) {
          chosen = b;
          break;
        }
        before += h->cnt[b];
      }
      s_before = before;
      s_prefix = prefix | ((uint32_t)chosen << shift);
    }
    __syncthreads();
  }
  const int idx = (int)s_prefix;
  __syncthreads();
  return idx;
}

// How many tokens of a tie group (n tokens of mass m each, `above` before
// them) the cumulative mass needs to reach the target.
__device__ __forceinline__ unsigned ties_needed(double above, unsigned n, double m, double target, bool strict) {
  if (n <= 1u || m <= 0.0) return 1u;
  const double k = (target - above) / (m / (double)n);
  if (!(k >= 0.0)) return 1u;
  if (k >= (double)n) return n;
  const unsigned r = strict ? (unsigned)floor(k) + 1u : (unsigned)ceil(k);
  return r < 1u ? 1u : r > n ? n : r;
}

__global__ void __launch_bounds__(kThreads) sample_kernel(const float* logits, int V, const float* temperature,
                                                           const float* top_p, const float* u, int32_t* out) {
  grid_dep_launch();
  grid_dep_wait();
  __shared__ Hist hist;
  __shared__ float red[33];
  __shared__ double red_d[33];
  __shared__ unsigned long long best_sh[32];
  const int b = blockIdx.x;
  const float* row = logits + (int64_t)b * V;
  const float T = temperature[b];
  if (!(T > 0.f)) {  // greedy: lowest index of the largest logit
    unsigned long long best = 0ull;
    for (int i = threadIdx.x; i < V; i += kThreads) {
      const unsigned long long k = argmax_key(row[i], (uint32_t)i);
      best = k > best ? k : best;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    if ((threadIdx.x & 31) == 0) best_sh[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long m = best_sh[0];
      for (int w = 1; w < kThreads / 32; ++w) m = best_sh[w] > m ? best_sh[w] : m;
      out[b] = (int32_t)argmax_key_index(m);
    }
    return;
  }
  const float sc = 1.4426950408889634f / T;  // log2(e) / T
  float mx = -3.402823466e38f;
  for (int i = threadIdx.x; i < V; i += kThreads) mx = fmaxf(mx, row[i]);
  const float lmax = block_max(mx, red);
  double z = 0.0;
  for (int i = threadIdx.x; i < V; i += kThreads) z += (double)exp2f((row[i] - lmax) * sc);
  const double Z = block_sum(z, red_d);
  // top-p cutoff: the first token whose cumulative probability reaches top_p
  const double tc = (double)top_p[b] * Z;
  const Quantile c = select_value(row, V, lmax, sc, tc, false, &hist);
  const unsigned rc = ties_needed(c.above, c.n_tie, c.m_tie, tc, false);
  const double z_kept = c.above + (c.n_tie > 0u ? c.m_tie / (double)c.n_tie : 0.0) * (double)rc;
  // the draw: the first token whose cumulative mass exceeds u * (kept mass)
  const double target = (double)u[b] * z_kept;
  const Quantile d = select_value(row, V, lmax, sc, target, true, &hist);
  unsigned rd = ties_needed(d.above, d.n_tie, d.m_tie, target, true);
  if (d.key == c.key && rd > rc) rd = rc;  // stay inside the kept set
  const int idx = d.n_tie <= 1u ? -1 : select_tie_index(row, V, d.key, rd, &hist);
  if (d.n_tie <= 1u) {  // the one token with this key
    __shared__ int s_idx;
    if (threadIdx.x == 0) s_idx = V;
    __syncthreads();
    for (int i = threadIdx.x; i < V; i += kThreads)
      if (float_order_key(row[i]) == d.key) atomicMin(&s_idx, i);
    __syncthreads();
    if (threadIdx.x == 0) out[b] = s_idx < V ? s_idx : 0;
    return;
  }
  if (threadIdx.x == 0) out[b] = idx;
}

}  // namespace smp

cudaError_t launch_sample(const float* logits, int batch, int V, const float* temperature, const float* top_p,
                          const float* u, int32_t* out, cudaStream_t s) {
  if (batch <= 0) return cudaSuccess;
  return launch_k(smp::sample_kernel, dim3(batch), dim3(smp::kThreads), 0, s, logits, V, temperature, top_p, u,
                  out);
}

}  // namespace tq
