// Prefill GEMM over the tiled Q4_0 / Q8_0 weights: Y[t][r] = sum_k W[r][k] X[t][k]
// for T tokens at once, so each weight unit is read once per 32 tokens instead of
// once per token.  Same exact operands and arithmetic as the decode GEMV
// (gemv_impl.cuh): codes as fp16 subnormals, the activations of every token as
// an fp16 hi/lo pair after a per-token power-of-two scale, mma.sync.m16n8k16
// with f32 sums, the block scale and the code-bias correction in f32.
//
// xprep_kernel turns the phase's input rows (optionally RMS-normalised with a
// gain, or silu(gate) * up) into the fragment table X[unit][token][block][128 B]
// plus the negated bias sums and the per-token output scale; unit-major order
// makes the 32 tokens of a CTA one contiguous copy per unit.
//
// qgemm_kernel: a CTA takes 8 tiles (128 rows) x 32 tokens and walks the K
// units (with few tokens, a 1/ks share of them: ks CTAs per tile group store
// partial sums and the last of them to finish adds the ks partials in split
// order); thread 0 streams each unit's 8 weight units, the tokens' fragments and
// bias sums into one of two shared-memory stages with 1-D bulk copies (bounded
// mbarrier waits).  Warp w multiplies tile w by the 32 tokens: per block the A
// fragment (rows g, g+8) is decoded once and used for the 8 groups of 4 tokens
// (the 8 B columns are the 4 tokens' hi and lo parts).  Prefill step of "Всередині
// LLM: чисте виконання на Python для Qwen3-0.6B на MLX" (steps 3-7 over all
// prompt positions).
#include "gemv_impl.cuh"

namespace tq {
namespace qg {

using gemv::half_of;
using gemv::lds128;
using gemv::mma16816;
using gemv::q4_operands;
using gemv::q8_operands;
using gemv::word_of;

constexpr int kTiles = 8;      // tiles (16 rows) per CTA
constexpr int kTok = 32;       // tokens per CTA
constexpr int kThreadsG = 256; // 8 warps, warp w <-> tile w
constexpr uint32_t kWaitLimitG = 1u << 22;

template <int WT>
struct QF {
  static constexpr int QU = unit_qs_bytes(WT);
  static constexpr int W = kTiles * (QU + kUnitD);          // weight units of one K step
  static constexpr int X = kTok * kUnitBlocks * 128;        // fragments of 32 tokens
  static constexpr int N = kTok * kUnitBlocks * 4;          // bias sums
  static constexpr int STAGE = W + X + N;
  static constexpr int SMEM = 2 * STAGE + 2 * 8;
};

// ------------------------------------------------------------------ xprep --

template <int WT>
__global__ void __launch_bounds__(256) xprep_kernel(const XPrepArgs a) {
  grid_dep_launch();
  grid_dep_wait();
  constexpr int PPT = 12288 / 8 / 256;  // pairs per thread at the largest K
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float sum_sh[8], max_sh[8];
  const int npairs = a.K / 8;
  const float* xr = a.x + (int64_t)t * a.ldx;
  const float* ur = a.up != nullptr ? a.up + (int64_t)t * a.ldx : nullptr;
  float4 v0[PPT], v1[PPT];
  float ss = 0.f, mx = 0.f;
#pragma unroll
  for (int r = 0; r < PPT; ++r) {
    const int pr = tid + r * 256;
    if (pr < npairs) {
      const int blk = pr >> 2, c = pr & 3;
      float4 p0 = *reinterpret_cast<const float4*>(xr + blk * 32 + 4 * c);
      float4 p1 = *reinterpret_cast<const float4*>(xr + blk * 32 + 16 + 4 * c);
      if (ur != nullptr) {  // silu(gate) * up
        const float4 u0 = *reinterpret_cast<const float4*>(ur + blk * 32 + 4 * c);
        const float4 u1 = *reinterpret_cast<const float4*>(ur + blk * 32 + 16 + 4 * c);
        p0 = make_float4(gemv::silu(p0.x) * u0.x, gemv::silu(p0.y) * u0.y, gemv::silu(p0.z) * u0.z,
                         gemv::silu(p0.w) * u0.w);
        p1 = make_float4(gemv::silu(p1.x) * u1.x, gemv::silu(p1.y) * u1.y, gemv::silu(p1.z) * u1.z,
                         gemv::silu(p1.w) * u1.w);
      }
      if (a.gain != nullptr) {
        ss = fmaf(p0.x, p0.x, fmaf(p0.y, p0.y, fmaf(p0.z, p0.z, fmaf(p0.w, p0.w, ss))));
        ss = fmaf(p1.x, p1.x, fmaf(p1.y, p1.y, fmaf(p1.z, p1.z, fmaf(p1.w, p1.w, ss))));
        const float4 g0 = *reinterpret_cast<const float4*>(a.gain + blk * 32 + 4 * c);
        const float4 g1 = *reinterpret_cast<const float4*>(a.gain + blk * 32 + 16 + 4 * c);
        p0 = make_float4(p0.x * g0.x, p0.y * g0.y, p0.z * g0.z, p0.w * g0.w);
        p1 = make_float4(p1.x * g1.x, p1.y * g1.y, p1.z * g1.z, p1.w * g1.w);
      }
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(p0.x), fabsf(p0.y)), fmaxf(fabsf(p0.z), fabsf(p0.w))));
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(p1.x), fabsf(p1.y)), fmaxf(fabsf(p1.z), fabsf(p1.w))));
      v0[r] = p0;
      v1[r] = p1;
    }
  }
  ss = warp_sum(ss);
  mx = warp_max(mx);
  if (lane == 0) {
    sum_sh[warp] = ss;
    max_sh[warp] = mx;
  }
  __syncthreads();
  ss = 0.f;
  mx = 0.f;
  for (int w = 0; w < 8; ++w) {
    ss += sum_sh[w];
    mx = fmaxf(mx, max_sh[w]);
  }
  const float scale = a.gain != nullptr ? 1.0f / sqrtf(ss / (float)a.K + a.eps) : 1.0f;
  mx *= scale;
  int e2 = 0;  // S = 2^e2 puts the largest |value| in [2^14, 2^15)
  if (mx > 0.f && mx <= 3.4e38f) e2 = 14 - (int)((__float_as_uint(mx) >> 23) & 0xffu) + 127;
  e2 = max(-100, min(126, e2));
  const float f = scale * __uint_as_float((uint32_t)(e2 + 127) << 23);
  if (tid == 0) a.inv_s[t] = __uint_as_float((uint32_t)(127 - e2) << 23) * 16777216.0f;  // 2^24 / S
#pragma unroll
  for (int r = 0; r < PPT; ++r) {
    const int pr = tid + r * 256;
    if (pr < npairs) {  // whole warps: npairs is a multiple of 32
      const int blk = pr >> 2, c = pr & 3;
      float e[8] = {v0[r].x * f, v0[r].y * f, v0[r].z * f, v0[r].w * f,
                    v1[r].x * f, v1[r].y * f, v1[r].z * f, v1[r].w * f};
      float bias = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
      bias *= WT == TQ_Q4_0 ? 8.0f : 128.0f;
      if (WT == TQ_Q4_0) {  // pairs (0,2) (1,3) (4,6)/16 (5,7)/16
        const float t1 = e[1], t5 = e[5];
        e[1] = e[2];
        e[2] = t1;
        e[4] *= 0.0625f;
        e[5] = e[6] * 0.0625f;
        e[6] = t5 * 0.0625f;
        e[7] *= 0.0625f;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float h0 = __uint_as_float(__float_as_uint(e[2 * k]) & 0xFFFFE000u);
        const float h1 = __uint_as_float(__float_as_uint(e[2 * k + 1]) & 0xFFFFE000u);
        const __half2 hh = __floats2half2_rn(h0, h1);
        const __half2 ll = __floats2half2_rn(e[2 * k] - h0, e[2 * k + 1] - h1);
        hi[k] = *reinterpret_cast<const uint32_t*>(&hh);
        lo[k] = *reinterpret_cast<const uint32_t*>(&ll);
      }
      bias += __shfl_xor_sync(0xffffffffu, bias, 1);
      bias += __shfl_xor_sync(0xffffffffu, bias, 2);
      const int u = blk / kUnitBlocks, j = blk % kUnitBlocks;
      const int64_t ent = ((int64_t)u * a.T + t) * kUnitBlocks + j;
      uint4* dst = reinterpret_cast<uint4*>(a.xtab + ent * 128);
      dst[c] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      dst[4 + c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      if (c == 0) a.xneg[ent] = -bias * 5.9604644775390625e-8f;  // 2^-24
    }
  }
}

// ------------------------------------------------------------------ GEMM --

struct TileMap {
  int T;         // tiles
  int tile0[4];  // first tile of each segment
  int row0[3];
};

__host__ __device__ inline TileMap tile_map(const QGemmArgs& a) {
  TileMap m;
  int t = 0, r = 0;
  for (int s = 0; s < 3; ++s) {
    m.tile0[s] = t;
    m.row0[s] = r;
    if (s < a.nseg) {
      t += (a.seg[s].rows + kTileRows - 1) / kTileRows;
      r += a.seg[s].rows;
    }
  }
  m.tile0[3] = t;
  m.T = t;
  return m;
}

__device__ __forceinline__ int seg_of(const TileMap& m, int t) {
  return t >= m.tile0[2] ? 2 : t >= m.tile0[1] ? 1 : 0;
}
__device__ __forceinline__ int sel3(const int (&v)[4], int s) { return s == 0 ? v[0] : s == 1 ? v[1] : v[2]; }
__device__ __forceinline__ int sel3r(const int (&v)[3], int s) { return s == 0 ? v[0] : s == 1 ? v[1] : v[2]; }

// Stage of K unit u: the weight units of the CTA's tiles (read-only: may be
// issued before the preceding kernel is done) and the tokens' fragments and
// bias sums; issue_weights arms the stage's barrier for both parts.
template <int WT>
__device__ __forceinline__ void issue_weights(const QGemmArgs& a, const TileMap& m, int tb, int ntok, int u, int G,
                                              uint8_t* st, uint64_t* bar) {
  using F = QF<WT>;
  uint32_t bytes = (uint32_t)(ntok * kUnitBlocks * (128 + 4));
  int nt = 0;
  for (int i = 0; i < kTiles; ++i)
    if (tb + i < m.T) ++nt;
  bytes += (uint32_t)(nt * (F::QU + kUnitD));
  mbar_arrive_expect_tx(bar, bytes);
  for (int i = 0; i < nt; ++i) {
    const int t = tb + i, s = seg_of(m, t);
    const int64_t off = (int64_t)(t - sel3(m.tile0, s)) * G + u;
    const GemvSeg& gs = a.seg[s];
    bulk_g2s(st + i * F::QU, gs.qs + off * F::QU, F::QU, bar);
    bulk_g2s(st + kTiles * F::QU + i * kUnitD, reinterpret_cast<const uint8_t*>(gs.d) + off * kUnitD, kUnitD, bar);
  }
}

template <int WT>
__device__ __forceinline__ void issue_x(const QGemmArgs& a, int t0, int ntok, int u, uint8_t* st, uint64_t* bar) {
  using F = QF<WT>;
  const int64_t ent = ((int64_t)u * a.T + t0) * kUnitBlocks;
  bulk_g2s(st + F::W, a.xtab + ent * 128, (uint32_t)(ntok * kUnitBlocks * 128), bar);
  bulk_g2s(st + F::W + F::X, a.xneg + ent, (uint32_t)(ntok * kUnitBlocks * 4), bar);
}

template <int WT>
__device__ __forceinline__ void issue_stage(const QGemmArgs& a, const TileMap& m, int tb, int t0, int ntok, int u,
                                            int G, uint8_t* st, uint64_t* bar) {
  issue_weights<WT>(a, m, tb, ntok, u, G, st, bar);
  issue_x<WT>(a, t0, ntok, u, st, bar);
}

// Q4_0: two CTAs per SM (128 registers; the two stages fit twice in shared
// memory), so each scheduler has four warps to hide latency with
template <int WT>
__global__ void __launch_bounds__(kThreadsG, WT == TQ_Q4_0 ? 2 : 1) qgemm_kernel(const __grid_constant__ QGemmArgs a) {
  using F = QF<WT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * F::STAGE);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const TileMap m = tile_map(a);
  const int G = a.K / 256;
  const int tb = blockIdx.x * kTiles, t0 = blockIdx.y * kTok;
  const int ntok = min(kTok, a.T - t0);
  const int ks = gridDim.z, z = blockIdx.z;
  const int ub = G * z / ks, ue = G * (z + 1) / ks;  // this CTA's K units
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_proxy_async();
  }
  __syncthreads();
  grid_dep_launch();
  // weights are read-only: the first two stages' units load while the
  // preceding kernel writes the fragment table
  if (tid == 0) {
    issue_weights<WT>(a, m, tb, ntok, ub, G, smem, &full[0]);
    if (ub + 1 < ue) issue_weights<WT>(a, m, tb, ntok, ub + 1, G, smem + F::STAGE, &full[1]);
  }
  grid_dep_wait();
  if (tid == 0) {
    issue_x<WT>(a, t0, ntok, ub, smem, &full[0]);
    if (ub + 1 < ue) issue_x<WT>(a, t0, ntok, ub + 1, smem + F::STAGE, &full[1]);
  }
  constexpr int NS = WT == TQ_Q4_0 ? 2 : 4;  // 16-byte code loads per row half
  const uint32_t sb = smem_addr(smem);
  float acc[8][2];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q][0] = acc[q][1] = 0.f;
  bool failed = false;
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  for (int u = ub; u < ue; ++u) {
    const int sidx = (u - ub) & 1;
    const bool ok = failed || mbar_wait_bounded(&full[sidx], (uint32_t)(((u - ub) >> 1) & 1), kWaitLimitG);
    if (!__all_sync(0xffffffffu, ok) && !failed) {
      if (lane == 0) set_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      failed = true;
    }
    const uint32_t st = sb + sidx * F::STAGE;
    const uint32_t qs = st + warp * F::QU, dq = st + kTiles * F::QU + warp * kUnitD;
    const uint32_t xs = st + F::W, xn = st + F::W + F::X;
    uint4 wv[2][NS], dv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int s = 0; s < NS; ++s) wv[h][s] = lds128(qs + ((h * NS + s) * 32 + lane) * 16);
      dv[h] = lds128(dq + (h * 8 + g) * 16);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t a0[4], a1[4];  // k-half 0 / 1 operands: rows g, g+8
      if (WT == TQ_Q4_0) {
        uint32_t g02, g13, gh02, gh13, e02, e13, eh02, eh13;
        q4_operands(word_of(wv[0][j >> 2], j & 3), g02, g13, gh02, gh13);
        q4_operands(word_of(wv[1][j >> 2], j & 3), e02, e13, eh02, eh13);
        a0[0] = g02; a0[1] = e02; a0[2] = g13; a0[3] = e13;
        a1[0] = gh02; a1[1] = eh02; a1[2] = gh13; a1[3] = eh13;
      } else {
        const uint4& r0 = wv[0][j >> 1];
        const uint4& r1 = wv[1][j >> 1];
        const int o = (j & 1) * 2;
        uint32_t g01, g23, e01, e23;
        q8_operands(word_of(r0, o), g01, g23);
        q8_operands(word_of(r1, o), e01, e23);
        a0[0] = g01; a0[1] = e01; a0[2] = g23; a0[3] = e23;
        q8_operands(word_of(r0, o + 1), g01, g23);
        q8_operands(word_of(r1, o + 1), e01, e23);
        a1[0] = g01; a1[1] = e01; a1[2] = g23; a1[3] = e23;
      }
      const float dg = half_bits_to_float(half_of(dv[0], j));
      const float dg8 = half_bits_to_float(half_of(dv[1], j));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        // lane (g, c): B column g = token 4q + g/2, part g%2 (hi, lo)
        const uint4 xf = lds128(xs + ((4 * q + (lane >> 3)) * kUnitBlocks + j) * 128 + (lane & 7) * 16);
        float cc[4];
        mma16816(cc, a0[0], a0[1], a0[2], a0[3], xf.x, xf.y, zero);
        mma16816(cc, a1[0], a1[1], a1[2], a1[3], xf.z, xf.w, cc);
        float nb;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(nb) : "r"(xn + ((4 * q + c) * kUnitBlocks + j) * 4));
        acc[q][0] = fmaf(dg, (cc[0] + cc[1]) + nb, acc[q][0]);
        acc[q][1] = fmaf(dg8, (cc[2] + cc[3]) + nb, acc[q][1]);
      }
    }
    __syncthreads();  // every warp is done with this stage
    if (tid == 0 && u + 2 < ue && !failed) issue_stage<WT>(a, m, tb, t0, ntok, u + 2, G, smem + sidx * F::STAGE, &full[sidx]);
  }
  // epilogue: lane (g, c) holds rows g, g+8 of tile tb + warp for tokens t0 + 4q + c
  const int t = tb + warp;
  const bool tile_ok = t < m.T;
  const int s = tile_ok ? seg_of(m, t) : 0;
  const int rows = a.seg[s].rows;
  if (ks > 1) {
    // this split's scaled sums, then the last split CTA of the tile group adds
    // all of them in split order
    if (tile_ok) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int tok = t0 + 4 * q + c;
        if (tok >= a.T) continue;
        const float is = a.inv_s[tok];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int local = (t - sel3(m.tile0, s)) * kTileRows + g + 8 * h;
          if (local < rows)
            a.part[((int64_t)z * a.T + tok) * a.ldy + sel3r(m.row0, s) + local] = acc[q][h] * is;
        }
      }
    }
    __shared__ int last_split;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      unsigned* ctr = a.counters + blockIdx.y * gridDim.x + blockIdx.x;
      last_split = atomicAdd(ctr, 1u) == (unsigned)(ks - 1);
      if (last_split) {
        *ctr = 0u;  // zero for the next launch
        __threadfence();
      }
    }
    __syncthreads();
    if (!last_split || !tile_ok) return;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int tok = t0 + 4 * q + c;
      if (tok >= a.T) continue;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int local = (t - sel3(m.tile0, s)) * kTileRows + g + 8 * h;
        if (local >= rows) continue;
        const int64_t o = (int64_t)tok * a.ldy + sel3r(m.row0, s) + local;
        float v = 0.f;
        for (int zz = 0; zz < ks; ++zz) v += __ldcg(a.part + (int64_t)zz * a.T * a.ldy + o);
        a.y[o] = a.residual != nullptr ? a.residual[o] + v : v;
      }
    }
    return;
  }
  if (tile_ok) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int tok = t0 + 4 * q + c;
      if (tok < a.T) {
        const float is = a.inv_s[tok];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int local = (t - sel3(m.tile0, s)) * kTileRows + g + 8 * h;
          if (local < rows) {
            const int64_t o = (int64_t)tok * a.ldy + sel3r(m.row0, s) + local;
            const float v = acc[q][h] * is;
            a.y[o] = a.residual != nullptr ? a.residual[o] + v : v;
          }
        }
      }
    }
  }
}

template <int WT>
cudaError_t launch_qgemm_t(const QGemmArgs& a, cudaStream_t s) {
  using F = QF<WT>;
  static PerDevice setup;
  int sms = 0;  // CTA slots: SMs x resident CTAs per SM
  cudaError_t e = per_device(setup, &sms, [](int dev, int& n) {
    cudaError_t r = cudaFuncSetAttribute(qgemm_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, F::SMEM);
    if (r != cudaSuccess) return r;
    int per = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kNumSMs;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, qgemm_kernel<WT>, kThreadsG, F::SMEM) != cudaSuccess ||
        per < 1)
      per = 1;
    n *= per;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const TileMap m = tile_map(a);
  dim3 grid((m.T + kTiles - 1) / kTiles, (a.T + kTok - 1) / kTok, 1);
  // Few tokens leave most SMs idle: split K so that waves x units per split
  // (plus a small cost per split for the partial sums) is least.
  const int G = a.K / 256, base = (int)(grid.x * grid.y);
  if (a.part != nullptr && a.counters != nullptr && base <= a.n_counters && base < 2 * sms) {
    double best = 1e30;
    for (int k = 1; k <= 16 && k <= G; ++k) {
      if (k > 1 && (int64_t)k * a.T * a.ldy > a.part_cap) break;
      const double cost = (double)((base * k + sms - 1) / sms) * ((G + k - 1) / k) + (k > 1 ? 0.1 * k : 0.0);
      if (cost < best) {
        best = cost;
        grid.z = k;
      }
    }
  }
  return launch_k(qgemm_kernel<WT>, grid, dim3(kThreadsG), F::SMEM, s, a);
}

}  // namespace qg

cudaError_t launch_xprep(int wtype, const XPrepArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.K % 256 != 0 || a.K > 12288) return cudaErrorInvalidValue;
  if (wtype == TQ_Q4_0) return launch_k(qg::xprep_kernel<TQ_Q4_0>, dim3(a.T), dim3(256), 0, s, a);
  return launch_k(qg::xprep_kernel<TQ_Q8_0>, dim3(a.T), dim3(256), 0, s, a);
}

cudaError_t launch_qgemm(int wtype, const QGemmArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.K % 256 != 0 || a.nseg < 1 || a.nseg > 3) return cudaErrorInvalidValue;
  return wtype == TQ_Q4_0 ? qg::launch_qgemm_t<TQ_Q4_0>(a, s) : qg::launch_qgemm_t<TQ_Q8_0>(a, s);
}

}  // namespace tq
