// Decode GEMV over Q4_0 / Q8_0 weights: y = W x with W stored as planar
// blocks of 32 along the input dimension, multiplied in f32 after exact
// in-register decoding (no activation quantization: "Inferencia local y
// arquitecturas", section "Elegir el motor").
//
// Pipeline (one CTA per SM).  One producer warp streams row tiles of the planar weights (the
// 16-byte nibble/byte chunks and the fp16 scales of a run of consecutive
// rows, both contiguous in HBM) into a ring of NS shared-memory stages with
// 1-D bulk copies through the TMA engine, completing on one mbarrier per
// stage; consumer warps release a stage through a second mbarrier as soon as
// they have read it.  Each CTA owns a contiguous range of rows, so the work is
// balanced to within one row, and the producer runs ahead of the consumers by
// up to NS stages (several tens of KB per SM in flight).
//
// Consumers.  A "team" of P threads covers one full row of K = 32*KPT*P
// inputs: thread t owns blocks t, t+P, ... of every row and keeps their
// activations in registers for the whole kernel.  A team takes R rows of each
// stage, reads each 16-byte chunk with one shared-memory load (consecutive
// threads, consecutive chunks: no bank conflicts), decodes it exactly and
// reduces the R row sums with a reduce-scatter butterfly (log2 R exchanges of
// halves, then a plain butterfly), finishing across warps in shared memory.
//
// Exact decoding.  A byte placed into the low byte of 0x4B000000 (one byte
// permute) reads as the float 2^23 + u.  Q4_0: low nibbles are masked in
// place (u = q), high nibbles are masked in place too (u = 16 q) and their
// activations are pre-scaled by 1/16 (exact); one packed f32x2 add of
// -(2^23 + 8) or -(2^23 + 128) yields q - 8 or 16 (q - 8) exactly.  Q8_0:
// codes are biased by 128 with one xor; -(2^23 + 128) yields q.  Packed f32x2
// FMAs then multiply by the activations, and the block's fp16 scale
// multiplies the block's partial sum.
//
// Fused prologue/epilogues: RMSNorm of x with a gain (step 3 of "Всередині
// LLM: чисте виконання на Python для Qwen3-0.6B на MLX"); residual add
// (step 7); SwiGLU over a gate/up pair (step 6); LM-head argmax with ties to
// the lowest index (step 8).
#pragma once

#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace tq {
namespace gemv {

constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

__device__ __forceinline__ float biased(uint32_t word, uint32_t sel) {
  return __uint_as_float(__byte_perm(word, 0x4B000000u, sel));
}

// sum_j x[j] (q_j - 8) for one Q4_0 block; x[16..31] hold x/16 (see above).
__device__ __forceinline__ float dot_q4(const uint4 w, const float* __restrict__ x) {
  const float2 blo = f2(-8388616.0f, -8388616.0f);  // -(2^23 + 8)
  const float2 bhi = f2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ws[i] & 0x0F0F0F0Fu;  // q of elements 4i .. 4i+3
    const uint32_t hi = ws[i] & 0xF0F0F0F0u;  // 16 q of elements 16+4i .. 16+4i+3
    const float2 a0 = __fadd2_rn(f2(biased(lo, 0x7650), biased(lo, 0x7651)), blo);
    const float2 a1 = __fadd2_rn(f2(biased(lo, 0x7652), biased(lo, 0x7653)), blo);
    const float2 b0 = __fadd2_rn(f2(biased(hi, 0x7650), biased(hi, 0x7651)), bhi);
    const float2 b1 = __fadd2_rn(f2(biased(hi, 0x7652), biased(hi, 0x7653)), bhi);
    acc0 = __ffma2_rn(f2(x[4 * i + 0], x[4 * i + 1]), a0, acc0);
    acc1 = __ffma2_rn(f2(x[4 * i + 2], x[4 * i + 3]), a1, acc1);
    acc0 = __ffma2_rn(f2(x[16 + 4 * i + 0], x[16 + 4 * i + 1]), b0, acc0);
    acc1 = __ffma2_rn(f2(x[16 + 4 * i + 2], x[16 + 4 * i + 3]), b1, acc1);
  }
  const float2 s = __fadd2_rn(acc0, acc1);
  return s.x + s.y;
}

// sum_j x[j] q_j over 16 int8 codes.
__device__ __forceinline__ float dot_q8_half(const uint4 w, const float* __restrict__ x) {
  const float2 bias = f2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = ws[i] ^ 0x80808080u;
    const float2 a0 = __fadd2_rn(f2(biased(u, 0x7650), biased(u, 0x7651)), bias);
    const float2 a1 = __fadd2_rn(f2(biased(u, 0x7652), biased(u, 0x7653)), bias);
    acc0 = __ffma2_rn(f2(x[4 * i + 0], x[4 * i + 1]), a0, acc0);
    acc1 = __ffma2_rn(f2(x[4 * i + 2], x[4 * i + 3]), a1, acc1);
  }
  const float2 s = __fadd2_rn(acc0, acc1);
  return s.x + s.y;
}

template <int R, int W>
__device__ __forceinline__ float reduce_scatter(float (&v)[R], int lane, int& slot) {
  int base = 0;
  int n = R;
#pragma unroll
  for (int o = W / 2; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < R / 2; ++i) {
        if (i < n / 2) {
          const float send = upper ? v[i] : v[i + n / 2];
          const float keep = upper ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      if (upper) base += n / 2;
      n /= 2;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  slot = base;
  return v[0];
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ void consumer_sync(int n_threads) {
  asm volatile("bar.sync 1, %0;" ::"r"(n_threads) : "memory");
}

// Shape of one instantiation.  The CTA (one per SM) has GROUPS groups of WPG
// consumer warps; each group streams its own contiguous share of the CTA's
// rows through its own ring of NS stages fed by its own producer lane.  A
// consumer warp owns R physical rows of every stage of its group (SwiGLU: R/2
// gate rows and the matching up rows) and sweeps the whole row: lane l takes
// blocks l, l+32, ... against the activations held in shared memory.
template <int WT_, int MODE_, int R_, int GROUPS_, int WPG_>
struct Shape {
  static constexpr int WT = WT_, MODE = MODE_, R = R_, GROUPS = GROUPS_, WPG = WPG_;
  static constexpr int CW = GROUPS * WPG;                 // consumer warps
  static constexpr int CT = CW * 32;
  static constexpr int THREADS = CT + 32;                 // + one producer warp
  static constexpr int CHUNK = WT == TQ_Q4_0 ? 16 : 32;   // qs bytes per block
  static constexpr int MATS = MODE == GEMV_SWIGLU ? 2 : 1;
  static constexpr int LR = R / MATS;                     // output rows per warp and stage
  static constexpr int SR = WPG * LR;                     // output rows per stage
};

// Runtime layout of the dynamic shared memory of one launch.
struct Layout {
  int nb, row_qs, row_d, stage_qs, stage, ns, off_x, off_bar, off_best, off_flag, bytes;
};

template <class S>
__host__ __device__ inline Layout layout_for(int K, int ns) {
  Layout L;
  auto up16 = [](int v) { return (v + 15) & ~15; };
  L.nb = K / 32;
  L.row_qs = L.nb * S::CHUNK;
  L.row_d = L.nb * 2;
  L.stage_qs = S::MATS * S::SR * L.row_qs;
  L.stage = L.stage_qs + ((S::MATS * S::SR * L.row_d + 127) / 128) * 128;
  L.ns = ns;
  L.off_x = S::GROUPS * ns * L.stage;
  L.off_bar = up16(L.off_x + ((K * 4 + 127) / 128) * 128);
  L.off_best = up16(L.off_bar + 2 * S::GROUPS * ns * 8);
  L.off_flag = up16(L.off_best + S::CW * 8 + S::CW * 4);
  L.bytes = L.off_flag + 16;
  return L;
}

// Row r of the concatenated segments -> (segment, row inside it, segment end).
__device__ __forceinline__ int seg_of(const GemvArgs& a, int r, int& local, int& seg_end) {
  int start = 0;
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    if (s < a.nseg) {
      const int end = start + a.seg[s].rows;
      if (r < end || s == a.nseg - 1) {
        local = r - start;
        seg_end = end;
        return s;
      }
      start = end;
    }
  }
  local = r;
  seg_end = a.N;
  return 0;
}

// 16-byte chunk c of block b of the activations lives at slot b*8 + (c ^ (b & 7)):
// lanes reading the same chunk of consecutive blocks hit distinct banks.
__device__ __forceinline__ int xslot(int b, int c) { return b * 8 + (c ^ (b & 7)); }

// Rows [begin, end) of the concatenated row space owned by group g of this CTA.
__device__ __forceinline__ void group_rows(int N, int groups, int g, int& begin, int& end) {
  const int64_t c0 = ((int64_t)N * blockIdx.x) / gridDim.x;
  const int64_t c1 = ((int64_t)N * (blockIdx.x + 1)) / gridDim.x;
  begin = (int)(c0 + ((c1 - c0) * g) / groups);
  end = (int)(c0 + ((c1 - c0) * (g + 1)) / groups);
}

template <class S>
__global__ void __launch_bounds__(S::THREADS, 1) gemv_kernel(const GemvArgs a, const int ns) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout L = layout_for<S>(a.K, ns);
  float4* xs = reinterpret_cast<float4*>(smem + L.off_x);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bar);  // [GROUPS][2][ns]
  unsigned long long* best_sh = reinterpret_cast<unsigned long long*>(smem + L.off_best);
  float* ssq = reinterpret_cast<float*>(smem + L.off_best + S::CW * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.off_flag);
  uint32_t* status = a.status;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nb = L.nb;

  if (tid == 0) {
    for (int s = 0; s < 2 * S::GROUPS * L.ns; ++s) mbar_init(&bars[s], (s / L.ns) % 2 == 0 ? 1 : S::WPG);
    *abort_flag = 0;
    fence_proxy_async();
  }
  __syncthreads();

  // The next kernel may start launching now: it only streams its own weights
  // until its consumers' grid_dep_wait().
  grid_dep_launch();

  if (warp == S::CW) {
    // ---------------------------------------------------------------- producer
    // Lane g feeds group g.  Weights are read-only: the stream starts before the
    // preceding kernel ends.
    if (lane >= S::GROUPS) return;
    const int g = lane;
    uint64_t* full = bars + (2 * g) * L.ns;
    uint64_t* empty = full + L.ns;
    int r_begin, r_end;
    group_rows(a.N, S::GROUPS, g, r_begin, r_end);
    uint8_t* ring = smem + g * L.ns * L.stage;
    int i = 0;
    for (int b = 0; b < a.B && !*abort_flag; ++b) {
      for (int r = r_begin; r < r_end && !*abort_flag;) {
        int local = r, seg_end = a.N, sg = 0;
        if (S::MODE != GEMV_SWIGLU) sg = seg_of(a, r, local, seg_end);
        const int n = min(S::SR, min(r_end - r, seg_end - r));
        const int stage = i % L.ns;
        if (i >= L.ns && !mbar_wait_bounded(&empty[stage], ((i / L.ns) - 1) & 1, kWaitLimit)) {
          set_status(status, TQ_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        uint8_t* st = ring + stage * L.stage;
        const uint32_t qbytes = (uint32_t)(n * L.row_qs), dbytes = (uint32_t)(n * L.row_d);
        mbar_arrive_expect_tx(&full[stage], S::MATS * (qbytes + dbytes));
#pragma unroll
        for (int m = 0; m < S::MATS; ++m) {
          const GemvSeg& gs = a.seg[S::MODE == GEMV_SWIGLU ? m : sg];
          bulk_g2s(st + m * S::SR * L.row_qs, gs.qs + (int64_t)local * L.row_qs, qbytes, &full[stage]);
          bulk_g2s(st + L.stage_qs + m * S::SR * L.row_d,
                   reinterpret_cast<const uint8_t*>(gs.d) + (int64_t)local * L.row_d, dbytes, &full[stage]);
        }
        r += n;
        ++i;
      }
    }
    // every issued copy lands before the CTA's shared memory is released
    for (int k = (i > L.ns ? i - L.ns : 0); k < i; ++k)
      mbar_wait_bounded(&full[k % L.ns], (k / L.ns) & 1, kWaitLimit);
    return;
  }

  // ------------------------------------------------------------------ consumers
  grid_dep_wait();  // activations, residual and outputs belong to earlier kernels
  constexpr int R = S::R;
  const int g = warp / S::WPG;
  const int wg = warp % S::WPG;
  uint64_t* full = bars + (2 * g) * L.ns;
  uint64_t* empty = full + L.ns;
  int r_begin, r_end;
  group_rows(a.N, S::GROUPS, g, r_begin, r_end);
  const uint8_t* ring = smem + g * L.ns * L.stage;
  int i = 0;
  for (int b = 0; b < a.B; ++b) {
    // activations -> shared memory (RMS-normalised, Q4_0 high halves scaled by 1/16)
    const float4* xg = reinterpret_cast<const float4*>(a.x + (int64_t)b * a.K);
    float scale = 1.0f;
    if (a.gain != nullptr) {
      float ss = 0.f;
      for (int q = tid; q < a.K / 4; q += S::CT) {
        const float4 v = xg[q];
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
      }
      ss = warp_sum(ss);
      if (lane == 0) ssq[warp] = ss;
      consumer_sync(S::CT);
      ss = 0.f;
      for (int w = 0; w < S::CW; ++w) ss += ssq[w];
      scale = 1.0f / sqrtf(ss / (float)a.K + a.eps);
    }
    for (int q = tid; q < a.K / 4; q += S::CT) {
      float4 v = xg[q];
      const int blk = q >> 3, c = q & 7;
      if (a.gain != nullptr) {
        const float4 gv = reinterpret_cast<const float4*>(a.gain)[q];
        v = make_float4(v.x * scale * gv.x, v.y * scale * gv.y, v.z * scale * gv.z, v.w * scale * gv.w);
      }
      if (S::WT == TQ_Q4_0 && c >= 4) v = make_float4(v.x * 0.0625f, v.y * 0.0625f, v.z * 0.0625f, v.w * 0.0625f);
      xs[xslot(blk, c)] = v;
    }
    consumer_sync(S::CT);

    unsigned long long best = 0ull;
    for (int r = r_begin; r < r_end;) {
      int local = r, seg_end = a.N;
      if (S::MODE != GEMV_SWIGLU) seg_of(a, r, local, seg_end);
      const int n = min(S::SR, min(r_end - r, seg_end - r));
      const int stage = i % L.ns;
      // Every lane waits (the warp sleeps in the barrier instead of one lane
      // spinning).  A timed-out wait sets the status and the abort flag; the
      // loop then runs to its end without waiting, on stale data, so that the
      // consumer barriers stay matched.
      bool ok = *abort_flag != 0 || mbar_wait_bounded(&full[stage], (i / L.ns) & 1, kWaitLimit);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          set_status(status, TQ_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
      }
      const uint8_t* st = ring + stage * L.stage;
      const uint16_t* dst = reinterpret_cast<const uint16_t*>(st + L.stage_qs);
      int srow[R];
      bool sval[R];
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int j = wg * S::LR + (S::MODE == GEMV_SWIGLU ? s / 2 : s);
        sval[s] = j < n;
        srow[s] = (S::MODE == GEMV_SWIGLU ? (s & 1) * S::SR : 0) + j;
      }
      float acc[R];
#pragma unroll
      for (int s = 0; s < R; ++s) acc[s] = 0.f;
      if (sval[0]) {
        for (int blk = lane; blk < nb; blk += 32) {
          float xr[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 v = xs[xslot(blk, c)];
            xr[4 * c] = v.x;
            xr[4 * c + 1] = v.y;
            xr[4 * c + 2] = v.z;
            xr[4 * c + 3] = v.w;
          }
#pragma unroll
          for (int s = 0; s < R; ++s) {
            if (sval[s]) {
              const float d = half_bits_to_float(dst[srow[s] * nb + blk]);
              const uint8_t* rowp = st + srow[s] * L.row_qs;
              if (S::WT == TQ_Q4_0) {
                const uint4 w = *reinterpret_cast<const uint4*>(rowp + blk * 16);
                acc[s] = fmaf(d, dot_q4(w, xr), acc[s]);
              } else {
                const uint4 w0 = *reinterpret_cast<const uint4*>(rowp + blk * 16);
                const uint4 w1 = *reinterpret_cast<const uint4*>(rowp + (nb + blk) * 16);
                acc[s] = fmaf(d, dot_q8_half(w0, xr) + dot_q8_half(w1, xr + 16), acc[s]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);

      int slot;
      const float v = reduce_scatter<R, 32>(acc, lane, slot);
      const bool writer = (lane % (32 / R)) == 0;
      if (S::MODE == GEMV_SWIGLU) {
        const float up = __shfl_down_sync(0xffffffffu, v, 32 / R);
        const int j = wg * S::LR + slot / 2;
        if (writer && (slot & 1) == 0 && j < n) a.y[(int64_t)b * a.N + r + j] = silu(v) * up;
      } else {
        const int j = wg * S::LR + slot;
        if (writer && j < n) {
          const int64_t o = (int64_t)b * a.N + r + j;
          if (S::MODE == GEMV_ARGMAX) {
            if (a.y != nullptr) a.y[o] = v;
            const unsigned long long key = argmax_key(v, (uint32_t)(r + j));
            best = key > best ? key : best;
          } else {
            a.y[o] = a.residual != nullptr ? a.residual[o] + v : v;
          }
        }
      }
      r += n;
      ++i;
    }

    if (S::MODE == GEMV_ARGMAX) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if (lane == 0) best_sh[warp] = best;
      consumer_sync(S::CT);
      if (tid == 0) {
        unsigned long long m = 0ull;
        for (int w = 0; w < S::CW; ++w) m = best_sh[w] > m ? best_sh[w] : m;
        if (m != 0ull) atomicMax(a.argmax_keys + b, m);
      }
    }
    consumer_sync(S::CT);  // x, ssq and best_sh are rewritten for the next token
  }
}

constexpr int kSmemMax = 220 * 1024;

template <class S>
int stages_for(int K) {
  for (int ns = 4; ns >= 1; --ns)
    if (layout_for<S>(K, ns).bytes <= kSmemMax) return ns;
  return 0;
}

template <class S>
cudaError_t launch(const GemvArgs& a, cudaStream_t s) {
  static int sms = 0;
  if (sms == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemMax);
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = kNumSMs;
  }
  const int ns = stages_for<S>(a.K);
  if (ns == 0) return cudaErrorInvalidValue;
  const Layout L = layout_for<S>(a.K, ns);
  int grid = a.N < sms ? a.N : sms;
  if (grid < 1) grid = 1;
  return launch_k(gemv_kernel<S>, dim3(grid), dim3(S::THREADS), L.bytes, s, a, ns);
}

}  // namespace gemv
}  // namespace tq
