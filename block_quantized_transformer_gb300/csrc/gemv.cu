// Decode GEMV over Q4_0 / Q8_0 weights: y = W x with W stored as planar
// blocks of 32 along the input dimension, multiplied in f32 after exact
// in-register decoding (no activation quantization: "Inferencia local y
// arquitecturas", section "Elegir el motor").
//
// Thread mapping.  A "team" of P threads covers one full row of K = 32*KPT*P
// inputs: thread t of the team owns blocks t, t+P, ..., t+(KPT-1)P of every
// row, keeps the matching 32*KPT activations in registers for the whole
// kernel, and streams one 16-byte chunk per block and row (one 128-bit load:
// a warp reads 512 contiguous bytes per instruction).  A team works on R rows
// at a time (R*KPT loads in flight per thread), reduces the R partial sums
// with a reduce-scatter butterfly (log2 R exchanges of halves, then a plain
// butterfly), and finishes across warps through shared memory when P > 32.
//
// Decoding: a nibble or byte is placed into the low byte of 0x4B000000 with
// one byte-permute, which reads as the float 2^23 + u; one packed f32x2 add
// of -(2^23 + 8) (Q4_0) or -(2^23 + 128) (Q8_0, codes biased by 128) yields
// the code exactly, and packed f32x2 FMAs multiply it by the activations.
// The block's fp16 scale multiplies the block's partial sum.
//
// Fused prologue/epilogues: RMSNorm of x (step 3 of "Всередині LLM ...
// Qwen3-0.6B на MLX") with a gain; residual add (step 7); SwiGLU over a
// gate/up pair (step 6); LM-head argmax with ties to the lowest index
// (step 8).
#include "kernels.cuh"

namespace tq {
namespace {

constexpr int TPB = 128;

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

__device__ __forceinline__ float byte_as_biased_float(uint32_t word, uint32_t sel) {
  return __uint_as_float(__byte_perm(word, 0x4B000000u, sel));
}

// sum_j x[j] * (q[j] - 8) over one Q4_0 block (16 nibble bytes in w).
__device__ __forceinline__ float dot_q4(const uint4 w, const float* __restrict__ x) {
  const float2 bias = f2(-8388616.0f, -8388616.0f);  // -(2^23 + 8)
  float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ws[i] & 0x0F0F0F0Fu;         // elements 4i .. 4i+3
    const uint32_t hi = (ws[i] >> 4) & 0x0F0F0F0Fu;  // elements 16+4i .. 16+4i+3
    float2 a0 = __fadd2_rn(f2(byte_as_biased_float(lo, 0x7650), byte_as_biased_float(lo, 0x7651)), bias);
    float2 a1 = __fadd2_rn(f2(byte_as_biased_float(lo, 0x7652), byte_as_biased_float(lo, 0x7653)), bias);
    float2 b0 = __fadd2_rn(f2(byte_as_biased_float(hi, 0x7650), byte_as_biased_float(hi, 0x7651)), bias);
    float2 b1 = __fadd2_rn(f2(byte_as_biased_float(hi, 0x7652), byte_as_biased_float(hi, 0x7653)), bias);
    acc0 = __ffma2_rn(f2(x[4 * i + 0], x[4 * i + 1]), a0, acc0);
    acc1 = __ffma2_rn(f2(x[4 * i + 2], x[4 * i + 3]), a1, acc1);
    acc0 = __ffma2_rn(f2(x[16 + 4 * i + 0], x[16 + 4 * i + 1]), b0, acc0);
    acc1 = __ffma2_rn(f2(x[16 + 4 * i + 2], x[16 + 4 * i + 3]), b1, acc1);
  }
  const float2 s = __fadd2_rn(acc0, acc1);
  return s.x + s.y;
}

// sum_j x[j] * q[j] over 16 int8 codes in w.
__device__ __forceinline__ float dot_q8_half(const uint4 w, const float* __restrict__ x) {
  const float2 bias = f2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = ws[i] ^ 0x80808080u;  // int8 q -> q + 128 in 0..255
    float2 a0 = __fadd2_rn(f2(byte_as_biased_float(u, 0x7650), byte_as_biased_float(u, 0x7651)), bias);
    float2 a1 = __fadd2_rn(f2(byte_as_biased_float(u, 0x7652), byte_as_biased_float(u, 0x7653)), bias);
    acc0 = __ffma2_rn(f2(x[4 * i + 0], x[4 * i + 1]), a0, acc0);
    acc1 = __ffma2_rn(f2(x[4 * i + 2], x[4 * i + 3]), a1, acc1);
  }
  const float2 s = __fadd2_rn(acc0, acc1);
  return s.x + s.y;
}

template <int WT>
struct Chunk;
template <>
struct Chunk<TQ_Q4_0> {
  uint4 q;
  uint16_t d;
};
template <>
struct Chunk<TQ_Q8_0> {
  uint4 q0, q1;
  uint16_t d;
};

template <int WT>
__device__ __forceinline__ void load_chunk(Chunk<WT>& c, const GemvSeg& s, int nb, int row, int blk);
template <>
__device__ __forceinline__ void load_chunk<TQ_Q4_0>(Chunk<TQ_Q4_0>& c, const GemvSeg& s, int nb,
                                                    int row, int blk) {
  const int64_t i = (int64_t)row * nb + blk;
  c.q = ldg_stream(s.qs + i * 16);
  c.d = ldg_u16(s.d + i);
}
template <>
__device__ __forceinline__ void load_chunk<TQ_Q8_0>(Chunk<TQ_Q8_0>& c, const GemvSeg& s, int nb,
                                                    int row, int blk) {
  const int64_t p0 = ((int64_t)row * 2) * nb + blk;
  c.q0 = ldg_stream(s.qs + p0 * 16);
  c.q1 = ldg_stream(s.qs + (p0 + nb) * 16);
  c.d = ldg_u16(s.d + (int64_t)row * nb + blk);
}

template <int WT>
__device__ __forceinline__ float dot_chunk(const Chunk<WT>& c, const float* x);
template <>
__device__ __forceinline__ float dot_chunk<TQ_Q4_0>(const Chunk<TQ_Q4_0>& c, const float* x) {
  return half_bits_to_float(c.d) * dot_q4(c.q, x);
}
template <>
__device__ __forceinline__ float dot_chunk<TQ_Q8_0>(const Chunk<TQ_Q8_0>& c, const float* x) {
  return half_bits_to_float(c.d) * (dot_q8_half(c.q0, x) + dot_q8_half(c.q1, x + 16));
}

// Reduce-scatter of R partial sums over W lanes (W a power of two <= 32,
// R <= W).  On return lane l holds the full sum of slot `slot`; lanes with
// (l % (W/R)) == 0 are the unique writers.
template <int R, int W>
__device__ __forceinline__ float reduce_scatter(float (&v)[R], int lane, int& slot) {
  float a[R];
#pragma unroll
  for (int i = 0; i < R; ++i) a[i] = v[i];
  int base = 0;
  int n = R;
#pragma unroll
  for (int o = W / 2; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < R / 2; ++i) {
        if (i < n / 2) {
          const float send = upper ? a[i] : a[i + n / 2];
          const float keep = upper ? a[i + n / 2] : a[i];
          a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      if (upper) base += n / 2;
      n /= 2;
    } else {
      a[0] += __shfl_xor_sync(0xffffffffu, a[0], o);
    }
  }
  slot = base;
  return a[0];
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

template <int WT, int KPT, int P, int R, int MODE>
__global__ void __launch_bounds__(TPB) gemv_kernel(const GemvArgs a) {
  constexpr int TEAMS = TPB / P;
  constexpr int W = P < 32 ? P : 32;    // lanes of one team inside a warp
  constexpr int WPT = P > 32 ? P / 32 : 1;  // warps per team
  constexpr int LOGICAL = MODE == GEMV_SWIGLU ? R / 2 : R;  // output rows per group

  __shared__ float red[2][TEAMS][WPT][R];
  __shared__ float ssq[TEAMS][WPT];
  __shared__ unsigned long long best_sh[TPB / 32];

  const int tid = threadIdx.x;
  const int team = tid / P;
  const int tl = tid % P;
  const int lane = tid & 31;
  const int wit = tl / 32;  // warp index inside the team
  const int K = a.K;
  const int nb = K / 32;
  const int n_groups = (a.N + LOGICAL - 1) / LOGICAL;

  for (int b = 0; b < a.B; ++b) {
    // ---- activations of this thread's blocks, optionally RMS-normalised
    float xr[KPT][32];
    const float* xb = a.x + (int64_t)b * K;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
      const float4* src = reinterpret_cast<const float4*>(xb + (tl + k * P) * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 v = src[j];
        xr[k][4 * j] = v.x;
        xr[k][4 * j + 1] = v.y;
        xr[k][4 * j + 2] = v.z;
        xr[k][4 * j + 3] = v.w;
      }
    }
    if (a.gain != nullptr) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < KPT; ++k)
#pragma unroll
        for (int j = 0; j < 32; ++j) ss = fmaf(xr[k][j], xr[k][j], ss);
#pragma unroll
      for (int o = W / 2; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (WPT > 1) {
        __syncthreads();
        if (lane == 0) ssq[team][wit] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int w = 0; w < WPT; ++w) ss += ssq[team][w];
      }
      const float inv = 1.0f / sqrtf(ss / (float)K + a.eps);
#pragma unroll
      for (int k = 0; k < KPT; ++k) {
        const float4* g = reinterpret_cast<const float4*>(a.gain + (tl + k * P) * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 gv = g[j];
          xr[k][4 * j] = xr[k][4 * j] * inv * gv.x;
          xr[k][4 * j + 1] = xr[k][4 * j + 1] * inv * gv.y;
          xr[k][4 * j + 2] = xr[k][4 * j + 2] * inv * gv.z;
          xr[k][4 * j + 3] = xr[k][4 * j + 3] * inv * gv.w;
        }
      }
    }

    unsigned long long best = 0ull;
    int round = 0;
    for (;; ++round) {
      const int g0 = (round * (int)gridDim.x + (int)blockIdx.x) * TEAMS;
      if (g0 >= n_groups) break;  // uniform across the CTA
      const int g = g0 + team;
      const bool active = g < n_groups;

      // ---- which matrix row each slot reads
      int srow[R], sseg[R];
      bool sval[R];
#pragma unroll
      for (int s = 0; s < R; ++s) {
        if (MODE == GEMV_SWIGLU) {
          const int r = g * LOGICAL + s / 2;
          sseg[s] = s & 1;
          srow[s] = r;
          sval[s] = active && r < a.N;
        } else {
          int r = g * R + s;
          sval[s] = active && r < a.N;
          int sg = 0;
          if (a.nseg > 1 && r >= a.seg[0].rows) {
            r -= a.seg[0].rows;
            sg = 1;
            if (a.nseg > 2 && r >= a.seg[1].rows) {
              r -= a.seg[1].rows;
              sg = 2;
            }
          }
          sseg[s] = sg;
          srow[s] = r;
        }
      }

      // ---- stream the R rows' chunks, then decode and multiply
      Chunk<WT> ch[R][KPT];
#pragma unroll
      for (int s = 0; s < R; ++s)
#pragma unroll
        for (int k = 0; k < KPT; ++k)
          if (sval[s]) load_chunk<WT>(ch[s][k], a.seg[sseg[s]], nb, srow[s], tl + k * P);
      float part[R];
#pragma unroll
      for (int s = 0; s < R; ++s) {
        part[s] = 0.f;
        if (sval[s]) {
#pragma unroll
          for (int k = 0; k < KPT; ++k) part[s] += dot_chunk<WT>(ch[s][k], xr[k]);
        }
      }

      // ---- reduce across the team
      int slot;
      float v = reduce_scatter<R, W>(part, lane, slot);
      const bool writer = (lane % (W / R)) == 0;
      if (WPT > 1) {
        if (writer) red[round & 1][team][wit][slot] = v;
        __syncthreads();
        if (wit == 0 && writer) {
          v = 0.f;
#pragma unroll
          for (int w = 0; w < WPT; ++w) v += red[round & 1][team][w][slot];
        }
      }
      const bool final_writer = writer && wit == 0;

      // ---- epilogue
      if (MODE == GEMV_SWIGLU) {
        // slot s+1 (up) lives W/R lanes above slot s (gate)
        float up = 0.f;
        if (WPT > 1) {
          if (final_writer && (slot & 1) == 0) {
#pragma unroll
            for (int w = 0; w < WPT; ++w) up += red[round & 1][team][w][slot + 1];
          }
        } else {
          up = __shfl_down_sync(0xffffffffu, v, W / R);
        }
        if (final_writer && (slot & 1) == 0 && active) {
          const int r = g * LOGICAL + slot / 2;
          if (r < a.N) a.y[(int64_t)b * a.N + r] = silu(v) * up;
        }
      } else if (final_writer && active) {
        const int r = g * R + slot;
        if (r < a.N) {
          const int64_t o = (int64_t)b * a.N + r;
          if (MODE == GEMV_ARGMAX) {
            if (a.y != nullptr) a.y[o] = v;
            const unsigned long long key = argmax_key(v, (uint32_t)r);
            best = key > best ? key : best;
          } else {
            a.y[o] = a.residual != nullptr ? a.residual[o] + v : v;
          }
        }
      }
    }

    if (MODE == GEMV_ARGMAX) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      __syncthreads();
      if (lane == 0) best_sh[tid / 32] = best;
      __syncthreads();
      if (tid == 0) {
        unsigned long long m = 0ull;
        for (int w = 0; w < TPB / 32; ++w) m = best_sh[w] > m ? best_sh[w] : m;
        if (m != 0ull) atomicMax(a.argmax_keys + b, m);
      }
    }
    if (a.B > 1) __syncthreads();
  }
}

__global__ void argmax_finish_kernel(const unsigned long long* keys, int n, int32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (int32_t)argmax_key_index(keys[i]);
}

// (KPT, P) such that K = 32 * KPT * P with P a power of two in [8, 128]
// preferring the largest P that is a multiple of 32 or the whole row.
bool pick_mapping(int K, int& kpt, int& p) {
  if (K % 32 != 0 || K <= 0) return false;
  const int nb = K / 32;
  const int cands[][2] = {{1, 128}, {3, 128}, {2, 128}, {1, 64}, {1, 32}, {3, 32}, {2, 32},
                          {4, 32},  {3, 64},  {2, 64},  {1, 16}, {1, 8},  {3, 8},  {2, 16},
                          {3, 16},  {2, 8},   {4, 8},   {4, 16}, {4, 64}, {4, 128}};
  for (auto& c : cands) {
    if (c[0] * c[1] == nb) {
      kpt = c[0];
      p = c[1];
      return true;
    }
  }
  return false;
}

template <int WT, int KPT, int P, int MODE>
cudaError_t launch_t(const GemvArgs& a, cudaStream_t s) {
  constexpr int R = KPT == 1 ? 8 : (KPT == 2 ? 4 : 2);
  constexpr int RR = (R > (P < 32 ? P : 32)) ? (P < 32 ? P : 32) : R;
  constexpr int TEAMS = TPB / P;
  constexpr int LOGICAL = MODE == GEMV_SWIGLU ? RR / 2 : RR;
  const int n_groups = (a.N + LOGICAL - 1) / LOGICAL;
  static int max_ctas = 0;
  if (max_ctas == 0) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<WT, KPT, P, RR, MODE>, TPB, 0);
    int dev = 0, sms = kNumSMs;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    max_ctas = (per_sm < 1 ? 1 : per_sm) * sms;
  }
  int grid = (n_groups + TEAMS - 1) / TEAMS;
  if (grid > max_ctas) grid = max_ctas;
  if (grid < 1) grid = 1;
  gemv_kernel<WT, KPT, P, RR, MODE><<<grid, TPB, 0, s>>>(a);
  return cudaGetLastError();
}

template <int WT, int MODE>
cudaError_t launch_wm(int kpt, int p, const GemvArgs& a, cudaStream_t s) {
#define TQ_CASE(KK, PP) \
  if (kpt == KK && p == PP) return launch_t<WT, KK, PP, MODE>(a, s);
  TQ_CASE(1, 128) TQ_CASE(3, 128) TQ_CASE(2, 128) TQ_CASE(4, 128)
  TQ_CASE(1, 64) TQ_CASE(2, 64) TQ_CASE(3, 64) TQ_CASE(4, 64)
  TQ_CASE(1, 32) TQ_CASE(2, 32) TQ_CASE(3, 32) TQ_CASE(4, 32)
  TQ_CASE(1, 16) TQ_CASE(2, 16) TQ_CASE(3, 16) TQ_CASE(4, 16)
  TQ_CASE(1, 8) TQ_CASE(2, 8) TQ_CASE(3, 8) TQ_CASE(4, 8)
#undef TQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

bool gemv_supported(int K) {
  int kpt, p;
  return pick_mapping(K, kpt, p);
}

cudaError_t launch_gemv(int wtype, int mode, const GemvArgs& a, cudaStream_t s) {
  int kpt, p;
  if (!pick_mapping(a.K, kpt, p)) return cudaErrorInvalidValue;
  if (a.N <= 0 || a.B <= 0) return cudaSuccess;
  if (wtype == TQ_Q4_0) {
    if (mode == GEMV_STORE) return launch_wm<TQ_Q4_0, GEMV_STORE>(kpt, p, a, s);
    if (mode == GEMV_SWIGLU) return launch_wm<TQ_Q4_0, GEMV_SWIGLU>(kpt, p, a, s);
    return launch_wm<TQ_Q4_0, GEMV_ARGMAX>(kpt, p, a, s);
  }
  if (mode == GEMV_STORE) return launch_wm<TQ_Q8_0, GEMV_STORE>(kpt, p, a, s);
  if (mode == GEMV_SWIGLU) return launch_wm<TQ_Q8_0, GEMV_SWIGLU>(kpt, p, a, s);
  return launch_wm<TQ_Q8_0, GEMV_ARGMAX>(kpt, p, a, s);
}

cudaError_t launch_argmax_finish(const unsigned long long* keys, int n, int32_t* out, cudaStream_t s) {
  argmax_finish_kernel<<<(n + 127) / 128, 128, 0, s>>>(keys, n, out);
  return cudaGetLastError();
}

}  // namespace tq
