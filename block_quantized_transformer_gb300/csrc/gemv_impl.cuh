// Decode GEMV over Q4_0 / Q8_0 weights, y = W x, with W in the tiled layout
// (kernels.cuh) and the products on the tensor cores.  The method multiplies
// f32 activations by the decoded weights, without quantizing the activations
// ("Inferencia local y arquitecturas", section "Elegir el motor"); here that
// product is formed as follows.
//
// Exact operands.  A code u read as the bits of an fp16 subnormal is exactly
// u * 2^-24: masking a word (one AND) yields the operand pairs, u = q for
// Q4_0 low nibbles, 16 q for the high nibbles (whose activations are pre-
// scaled by 1/16), u = q + 128 for Q8_0 (codes biased with one xor).  The
// activation vector, scaled by a power of two S so that its largest
// magnitude lies in [2^14, 2^15), is carried as an unevaluated sum hi + lo of
// two fp16 values (hi = v with its low 13 mantissa bits cleared, lo =
// fp16(v - hi)), which keeps 21 significant bits.  mma.sync.m16n8k16
// multiplies the 16 x 16 weight fragment by the columns (hi, lo): every
// product is exact in f32 and the tensor core sums in f32.  The code bias
// (8 for Q4_0, 128 for Q8_0) times the block's sum of activations, computed
// once per block for all rows, is subtracted from the block's sum, the
// block's fp16 scale multiplies it in an f32 FMA, and the row total is
// multiplied by 2^24 / S (exact).
//
// Work split.  The units (16 rows x 256 inputs) of a GEMV are numbered tile
// by tile; every CTA (one per SM) takes a contiguous range of whole tiles,
// and every consumer warp a contiguous sub-range of the CTA's units.  A warp
// sums each of its tiles in registers; a tile it covers whole is finished by
// that warp, a tile shared with other warps is summed from their partials in
// warp order after a CTA barrier.  The order of every sum is fixed, so
// results do not depend on timing.  (Splitting tiles between CTAs balances
// bytes better but costs a grid-wide reduction per tile at the end of every
// phase, which measured slower.)
//
// Pipeline.  Every consumer warp reads its units from its own ring of shared-
// memory slots, which a lane of one of kP producer warps fills with 1-D bulk
// copies through the TMA engine (full/empty mbarriers, every wait bounded).
// A bulk-copy issue can stall on a full TMA queue; only a producer waits then.
//
// Chains.  One launch runs up to kMaxPhases GEMVs in a row; CTAs meet at a
// grid-wide counter between phases (the next phase reads what the previous
// one wrote), while every warp's ring already holds the first units of its
// next phase, so the weight stream does not drain at phase boundaries.
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
constexpr uint32_t kSyncLimit = 1u << 24;
#ifndef TQ_GEMV_CONSUMER_WARPS
#define TQ_GEMV_CONSUMER_WARPS 8
#endif
#ifndef TQ_GEMV_SLOT_UNITS_Q4
#define TQ_GEMV_SLOT_UNITS_Q4 4
#endif
constexpr int kW = TQ_GEMV_CONSUMER_WARPS;  // consumer warps
constexpr int kCT = kW * 32;            // consumer threads
#ifndef TQ_GEMV_PRODUCER_WARPS
#define TQ_GEMV_PRODUCER_WARPS 4  // a bulk-copy issue can stall; four issuers keep more copies in flight
#endif
constexpr int kP = TQ_GEMV_PRODUCER_WARPS;  // producer warps
constexpr int kThreads = kCT + 32 * kP;
constexpr int kSmemMax = 227 * 1024;
constexpr int kXBlockBytes = 128;       // fp16 hi/lo fragments of one 32-input block
constexpr int kMaxK = 12288;
constexpr int kPPT = (kMaxK / 8 + kCT - 1) / kCT;  // activation pairs per thread, at most

// A ring slot holds SU units of one matrix (SU/2 of a gate/up pair); each
// matrix's run of units arrives in two bulk copies (codes, scales), so a
// copy moves several KB: the TMA engine's cost per copy then stays small
// against its cost per byte.
template <int WT>
struct Fmt {
  static constexpr int QU = unit_qs_bytes(WT);       // code bytes of a unit
  static constexpr int UB = QU + kUnitD;             // unit bytes
  static constexpr int SU = nib4(WT) ? TQ_GEMV_SLOT_UNITS_Q4 : 2;  // units per slot (even)
  static constexpr int SLOT = SU * UB;
};

// ------------------------------------------------------------ tensor core --

// D = A B + C, A 16x16 fp16 (row), B 16x8 fp16 (col), C/D f32.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint16_t half_of(const uint4& v, int j) {
  const uint32_t w = word_of(v, j >> 1);
  return (uint16_t)((j & 1) ? (w >> 16) : (w & 0xffffu));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Exact fp16 operand pairs (u * 2^-24) of one code word (see the header
// comment).  Q4_0 word c of a block: bytes 4c..4c+3 hold inputs 4c..4c+3
// (low nibbles) and 16+4c..19+4c (high nibbles).  Out: k-half 0
// {(4c,4c+2), (4c+1,4c+3)} as q, k-half 1 {(16+4c,18+4c), (17+4c,19+4c)}
// as 16 q.
__device__ __forceinline__ void q4_operands(uint32_t w, uint32_t& l02, uint32_t& l13, uint32_t& h02,
                                            uint32_t& h13) {
  const uint32_t w8 = w >> 8;
  l02 = w & 0x000F000Fu;
  l13 = w8 & 0x000F000Fu;
  h02 = w & 0x00F000F0u;
  h13 = w8 & 0x00F000F0u;
}

// Q8_0 word i of a block (codes 4i..4i+3): pairs (4i, 4i+1), (4i+2, 4i+3) as
// q + 128.
__device__ __forceinline__ void q8_operands(uint32_t w, uint32_t& p01, uint32_t& p23) {
  const uint32_t u = w ^ 0x80808080u;
  p01 = __byte_perm(u, 0u, 0x4140);
  p23 = __byte_perm(u, 0u, 0x4342);
}

// Sum of one unit (16 rows x 8 blocks) of MATS matrices into acc[m][0] (row g
// of the tile) and acc[m][1] (row g + 8); lane = 4 g + c.  qs/dq: shared
// addresses of the units' codes and scales (matrix m at + m * mstride_q / _d),
// xt / xn: shared addresses of the x fragments and of the negated bias sums
// of the unit's first block (the operands carry the biased codes, so a
// block's tensor-core sum exceeds the wanted sum by bias * sum(x) * 2^-24,
// which the prologue computed once for all rows).  AFFINE4: the operands are
// the plain codes q, the prologue's table holds -sum(x) * 2^-24 per block,
// and a block adds s * (its sum) + b * sum(x) with its group's bf16 s and b.
template <int WT, int MATS>
__device__ __forceinline__ void unit_dot(uint32_t qs, uint32_t mstride_q, uint32_t dq, uint32_t mstride_d,
                                         uint32_t xt, uint32_t xn, int lane, float (&acc)[MATS][2]) {
  constexpr int NS = nib4(WT) ? 2 : 4;  // 16-byte code loads per row half
  const int g = lane >> 2;
  uint4 wv[MATS][2][NS];
  uint4 dv[MATS][2];
#pragma unroll
  for (int m = 0; m < MATS; ++m) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int s = 0; s < NS; ++s) wv[m][h][s] = lds128(qs + m * mstride_q + ((h * NS + s) * 32 + lane) * 16);
      dv[m][h] = lds128(dq + m * mstride_d + (h * 8 + g) * 16);
    }
  }
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  const uint4 nbv[2] = {lds128(xn), lds128(xn + 16)};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float nb = __uint_as_float(word_of(nbv[j >> 2], j & 3));
    uint4 xf = make_uint4(0u, 0u, 0u, 0u);  // lanes 0-3: hi column, 4-7: lo column, others zero
    if (lane < 8) xf = lds128(xt + j * kXBlockBytes + lane * 16);
#pragma unroll
    for (int m = 0; m < MATS; ++m) {
      float c[4];
      if (nib4(WT)) {
        uint32_t g02, g13, gh02, gh13, e02, e13, eh02, eh13;
        q4_operands(word_of(wv[m][0][j >> 2], j & 3), g02, g13, gh02, gh13);
        q4_operands(word_of(wv[m][1][j >> 2], j & 3), e02, e13, eh02, eh13);
        mma16816(c, g02, e02, g13, e13, xf.x, xf.y, zero);
        mma16816(c, gh02, eh02, gh13, eh13, xf.z, xf.w, c);
      } else {
        const uint4& r0 = wv[m][0][j >> 1];
        const uint4& r1 = wv[m][1][j >> 1];
        const int o = (j & 1) * 2;
        uint32_t g01, g23, e01, e23;
        q8_operands(word_of(r0, o), g01, g23);
        q8_operands(word_of(r1, o), e01, e23);
        mma16816(c, g01, e01, g23, e23, xf.x, xf.y, zero);
        q8_operands(word_of(r0, o + 1), g01, g23);
        q8_operands(word_of(r1, o + 1), e01, e23);
        mma16816(c, g01, e01, g23, e23, xf.z, xf.w, c);
      }
      if (WT == TQ_AFFINE4) {  // group j / 2: (s, b) at elements 2 (j / 2), + 1
        const int e = j & ~1;
        acc[m][0] = fmaf(bf16_bits_to_float(half_of(dv[m][0], e)), c[0] + c[1],
                         fmaf(-bf16_bits_to_float(half_of(dv[m][0], e + 1)), nb, acc[m][0]));
        acc[m][1] = fmaf(bf16_bits_to_float(half_of(dv[m][1], e)), c[2] + c[3],
                         fmaf(-bf16_bits_to_float(half_of(dv[m][1], e + 1)), nb, acc[m][1]));
      } else {
        acc[m][0] = fmaf(half_bits_to_float(half_of(dv[m][0], j)), (c[0] + c[1]) + nb, acc[m][0]);
        acc[m][1] = fmaf(half_bits_to_float(half_of(dv[m][1], j)), (c[2] + c[3]) + nb, acc[m][1]);
      }
    }
  }
}

// ------------------------------------------------------------- geometry --

// Per-phase work geometry, computed the same way by every thread.
struct Geo {
  int G;        // units per tile row (K / 256)
  int T;        // tiles
  int U;        // units = T * G
  int mats;     // 2 for SWIGLU (gate, up), else 1
  int k;        // units per ring slot
  int Cp;       // CTAs with work
  int tile0[4]; // first tile of each segment; tile0[nseg] = T
  int row0[3];  // first output row of each segment
};

__host__ __device__ inline Geo geo_of(const GemvArgs& a, int mode, int grid, int su) {
  Geo q;
  q.G = a.K / 256;
  q.mats = mode == GEMV_SWIGLU ? 2 : 1;
  q.k = mode == GEMV_SWIGLU ? su / 2 : su;
  const int nseg = mode == GEMV_SWIGLU ? 1 : a.nseg;
  int t = 0, r = 0;
  for (int s = 0; s < 3; ++s) {
    q.tile0[s] = t;
    q.row0[s] = r;
    if (s < nseg) {
      const int rows = mode == GEMV_SWIGLU ? a.N : a.seg[s].rows;
      t += (rows + kTileRows - 1) / kTileRows;
      r += rows;
    }
  }
  q.tile0[3] = t;
  q.T = t;
  q.U = t * q.G;
  q.Cp = grid < q.T ? grid : q.T;
  if (q.Cp < 1) q.Cp = 1;
  return q;
}

__device__ __forceinline__ void cta_range(const Geo& q, int c, int& u0, int& u1) {
  if (c >= q.Cp) {
    u0 = u1 = q.U;
  } else {
    u0 = q.G * (int)((int64_t)q.T * c / q.Cp);
    u1 = q.G * (int)((int64_t)q.T * (c + 1) / q.Cp);
  }
}

__device__ __forceinline__ void warp_range(int u0, int u1, int w, int& a, int& b) {
  const int n = u1 - u0;
  a = u0 + (int)((int64_t)n * w / kW);
  b = u0 + (int)((int64_t)n * (w + 1) / kW);
}

__device__ __forceinline__ int seg_of_tile(const Geo& q, int t) {
  return t >= q.tile0[2] ? 2 : t >= q.tile0[1] ? 1 : 0;
}

// q.tile0[s] / q.row0[s] with constant indices only (no local-memory copy)
__device__ __forceinline__ int seg_tile0(const Geo& q, int s) {
  return s == 0 ? q.tile0[0] : s == 1 ? q.tile0[1] : q.tile0[2];
}
__device__ __forceinline__ int seg_row0(const Geo& q, int s) {
  return s == 0 ? q.row0[0] : s == 1 ? q.row0[1] : q.row0[2];
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory"); }


// Final value(s) of row rr of tile t: scale, epilogue, store.  resid: this
// CTA's residual rows from tile t0 on, prefetched to shared memory, or null;
// keep: the stored value also replaces the residual row in shared memory (a
// later phase of the chain adds to the same rows).
__device__ __forceinline__ void finish_row(const GemvArgs& a, int mode, const Geo& q, int b, int t, int rr,
                                           float v, float up, float* resid, bool keep, int t0, float inv_s,
                                           unsigned long long& best) {
  const int s = seg_of_tile(q, t);
  const int local = (t - seg_tile0(q, s)) * kTileRows + rr;
  const int rows = mode == GEMV_SWIGLU ? a.N : a.seg[s].rows;
  if (local >= rows) return;
  const int row = seg_row0(q, s) + local;
  const int64_t o = (int64_t)b * a.N + row;
  v *= inv_s;
  if (mode == GEMV_SWIGLU) {
    a.y[o] = gate_act(v, a.act) * (up * inv_s);
  } else if (mode == GEMV_ARGMAX) {
    if (a.softcap > 0.f) v = a.softcap * tanhf(v / a.softcap);
    if (a.y != nullptr) a.y[o] = v;
    const unsigned long long key = argmax_key(v, (uint32_t)row);
    best = key > best ? key : best;
  } else {
    const float r = a.residual == nullptr ? 0.f
                    : resid != nullptr ? resid[(t - t0) * kTileRows + rr]
                                       : __ldcg(a.residual + o);
    const float yv = a.bias != nullptr ? (r + v) + a.bias[row] : r + v;
    a.y[o] = yv;
    if (keep) resid[(t - t0) * kTileRows + rr] = yv;
  }
}

// A warp's sums of tile t: finished here when the warp covers the whole tile,
// else kept as a partial (slot 0: the warp's first tile, 1: its last).
__device__ __forceinline__ void flush_tile(const GemvArgs& a, int mode, const Geo& q, int b, int t, int wa,
                                           int wb, int warp, int lane, const float (&acc)[2][2], float* red,
                                           float* resid, bool keep, int t0, float inv_s,
                                           unsigned long long& best) {
  const int g = lane >> 2;
  if ((lane & 3) != 0) return;
  if (t * q.G >= wa && t * q.G + q.G <= wb) {
    finish_row(a, mode, q, b, t, g, acc[0][0], acc[1][0], resid, keep, t0, inv_s, best);
    finish_row(a, mode, q, b, t, g + 8, acc[0][1], acc[1][1], resid, keep, t0, inv_s, best);
  } else {
    float* r = red + (warp * 2 + (t == wa / q.G ? 0 : 1)) * 32;
    r[g] = acc[0][0];
    r[g + 8] = acc[0][1];
    r[16 + g] = acc[1][0];
    r[16 + g + 8] = acc[1][1];
  }
}

// Tile t shared between warps of this CTA, summed by its first contributing
// warp from the partials in warp order.  Lane r < 16 ends with row r (lanes
// 16-31: the up rows of SWIGLU).
__device__ __forceinline__ void reduce_tile(const GemvArgs& a, int mode, const Geo& q, int b, int t, int u0, int u1,
                                            int warp, int lane, const float* red, float* resid, bool keep, int t0,
                                            float inv_s, unsigned long long& best) {
  const int te = min(t * q.G + q.G, u1);
  float v = 0.f;
  for (int w = warp; w < kW; ++w) {
    int xa, xe;
    warp_range(u0, u1, w, xa, xe);
    if (xa >= xe) continue;
    if (xa >= te) break;
    v += red[(w * 2 + (t == xa / q.G ? 0 : 1)) * 32 + lane];
  }
  const float up = __shfl_down_sync(0xffffffffu, v, 16);
  if (lane < 16) finish_row(a, mode, q, b, t, lane, v, up, resid, keep, t0, inv_s, best);
}

// ---------------------------------------------------------------- layout --

constexpr int kResidTiles = 64;  // residual rows prefetched to shared memory (tiles per CTA)
constexpr int kResidPerThread = (kResidTiles * kTileRows + kCT - 1) / kCT;

struct Smem {
  int ring, xtab, xneg, red, resid, misc, bars, bytes;
};

__host__ __device__ inline Smem smem_layout(int slot, int depth, int max_k) {
  Smem L;
  L.ring = 0;
  L.xtab = kW * depth * slot;
  L.xneg = L.xtab + (max_k / 32) * kXBlockBytes;  // negated bias sum per block
  L.red = L.xneg + (max_k / 32) * 4;
  L.resid = L.red + kW * 2 * 32 * 4;             // partial tile sums [warp][2][32]
  L.misc = L.resid + kResidTiles * kTileRows * 4;
  L.bars = L.misc + kW * 8 + kW * 4 * 2 + 16;    // best keys, sums, maxima, flag
  L.bars = (L.bars + 15) & ~15;
  L.bytes = L.bars + kW * depth * 2 * 8;
  return L;
}

// The slot sequence of one warp over all phases and tokens of a chain.  The
// warp's prefetch cursor walks it up to `depth` slots ahead of the warp's
// consumption.  Every lane keeps the same cursor; lane 0 issues the copies.
struct Cursor {
  int p, b, u, wa, wb;
  Geo q;
};

template <int WT>
__device__ __forceinline__ void cursor_enter(Cursor& cu, const GemvChain& ch, int cta, int C, int w) {
  for (; cu.p < ch.n; ++cu.p) {
    const GemvArgs& a = ch.ph[cu.p];
    cu.q = geo_of(a, ch.mode[cu.p], C, Fmt<WT>::SU);
    int u0, u1;
    cta_range(cu.q, cta, u0, u1);
    warp_range(u0, u1, w, cu.wa, cu.wb);
    cu.b = 0;
    cu.u = cu.wa;
    if (cu.wa < cu.wb) return;
  }
}

// Copy the cursor's next slot into `st` (completing on `bar`) and advance.
template <int WT>
__device__ __forceinline__ void cursor_issue(Cursor& cu, const GemvChain& ch, int cta, int C, int w,
                                             uint8_t* st, uint64_t* bar) {
  using F = Fmt<WT>;
  const GemvArgs& a = ch.ph[cu.p];
  const int mode = ch.mode[cu.p];
  const Geo& q = cu.q;
  const int t = cu.u / q.G;
  const int n = min(q.k, min((t + 1) * q.G, cu.wb) - cu.u);
  {
    mbar_arrive_expect_tx(bar, (uint32_t)(q.mats * n * F::UB));
    const int s = seg_of_tile(q, t);
    const int64_t off = (int64_t)(t - seg_tile0(q, s)) * q.G + (cu.u - t * q.G);  // unit inside the segment
    for (int m = 0; m < q.mats; ++m) {
      const GemvSeg& gs = a.seg[mode == GEMV_SWIGLU ? m : s];
      bulk_g2s(st + m * q.k * F::QU, gs.qs + off * F::QU, (uint32_t)(n * F::QU), bar);
      bulk_g2s(st + q.mats * q.k * F::QU + m * q.k * kUnitD, reinterpret_cast<const uint8_t*>(gs.d) + off * kUnitD,
               (uint32_t)(n * kUnitD), bar);
    }
  }
  cu.u += n;
  if (cu.u >= cu.wb) {
    cu.u = cu.wa;
    if (++cu.b >= a.B) {
      ++cu.p;
      cursor_enter<WT>(cu, ch, cta, C, w);
    }
  }
}

template <int WT>
__global__ void __launch_bounds__(kThreads, 1) gemv_chain_kernel(const __grid_constant__ GemvChain ch,
                                                                 const int depth, const int max_k) {
  using F = Fmt<WT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const Smem L = smem_layout(F::SLOT, depth, max_k);
  const uint32_t sbase = smem_addr(smem);
  float* red = reinterpret_cast<float*>(smem + L.red);
  unsigned long long* best_sh = reinterpret_cast<unsigned long long*>(smem + L.misc);
  float* sum_sh = reinterpret_cast<float*>(smem + L.misc + kW * 8);
  float* max_sh = sum_sh + kW;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + kW * 8 + kW * 8);
  uint32_t* status = ch.ph[0].status;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, C = gridDim.x;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);  // [warp][full/empty][depth]

  if (tid == 0) {
    for (int k = 0; k < kW * 2 * depth; ++k) mbar_init(&bars[k], 1);
    *abort_flag = 0;
    fence_proxy_async();
  }
  __syncthreads();
  // A chain's CTAs meet at grid-wide counters, so every CTA must be resident
  // before a later kernel may take an SM: with several phases the dependent
  // launch is released only after the first counter is full (every CTA is
  // running); a single GEMV releases it at once.
  if (ch.n == 1) grid_dep_launch();

  if (warp >= kW) {
    // ---------------------------------------------------------------- producer
    // Lane l of producer warp pw keeps consumer warp pw + kP l's ring full: in
    // a loop common to the lanes, every lane whose next stage is free (non-
    // blocking test) issues that slot's copies, so a ring that is still being
    // read never holds up the others, and a bulk-copy issue that stalls on a
    // full TMA queue stalls only a producer.  Weights are read-only: nothing here waits for other
    // kernels or other CTAs, so the first slots load while the consumers wait
    // for the kernel that writes this launch's activations.
    const int pw = warp - kW;                 // producer warp pw serves rings pw, pw + kP, ...
    const bool mine = pw + kP * lane < kW;
    const int w = mine ? pw + kP * lane : 0;
    uint64_t* full = bars + w * 2 * depth;
    uint64_t* empty = full + depth;
    uint8_t* ring = smem + L.ring + w * depth * F::SLOT;
    Cursor cu;
    cu.p = mine ? 0 : ch.n;
    cursor_enter<WT>(cu, ch, cta, C, w);
    int issued = 0;
    uint32_t idle = 0;
    while (true) {
      const bool more = cu.p < ch.n && !*abort_flag;
      if (!__any_sync(0xffffffffu, more)) break;
      bool did = false;
      if (more) {
        const int stage = issued % depth;
        if (issued < depth || mbar_test_wait(&empty[stage], ((issued / depth) - 1) & 1)) {
          cursor_issue<WT>(cu, ch, cta, C, w, ring + stage * F::SLOT, &full[stage]);
          ++issued;
          did = true;
        }
      }
      if (__any_sync(0xffffffffu, did)) {
        idle = 0;
      } else if (++idle > kWaitLimit) {  // no consumer released a stage for a long time
        if (lane == 0) {
          set_status(status, TQ_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      } else if (idle > 64) {
        __nanosleep(32);
      }
    }
    // every issued copy lands before the CTA's shared memory is released
    if (mine)
      for (int k = (issued > depth ? issued - depth : 0); k < issued; ++k)
        mbar_wait_bounded(&full[k % depth], (k / depth) & 1, kWaitLimit);
    return;
  }

  // ------------------------------------------------------------------ consumers
  uint64_t* full = bars + warp * 2 * depth;
  uint64_t* empty = full + depth;

  const uint32_t ring_s = sbase + L.ring + warp * depth * F::SLOT;
  const uint32_t xtab = sbase + L.xtab, xneg = sbase + L.xneg;
  int i = 0;  // slots consumed
  // Phase 0 (output projection) and phase 2 (down projection) both add to the
  // residual stream: with one token, the same output rows and hence the same
  // tiles per CTA, phase 0's results are phase 2's residual rows.
  const bool carry = ch.n > 2 && ch.mode[0] == GEMV_STORE && ch.mode[2] == GEMV_STORE && ch.ph[0].B == 1 &&
                     ch.ph[2].B == 1 && ch.ph[0].nseg == 1 && ch.ph[2].nseg == 1 &&
                     ch.ph[0].residual != nullptr && ch.ph[2].residual == ch.ph[0].y && ch.ph[2].N == ch.ph[0].N &&
                     ch.ph[0].y != nullptr;
  for (int p = 0; p < ch.n; ++p) {
    const GemvArgs& a = ch.ph[p];
    const int mode = ch.mode[p];
    const Geo q = geo_of(a, mode, C, Fmt<WT>::SU);
    int u0, u1, wa, wb;
    cta_range(q, cta, u0, u1);
    warp_range(u0, u1, warp, wa, wb);
    // wait for the producers of this phase's activations
    if (p == 0) {
      grid_dep_wait();
    } else {
      if (tid == 0 && !*abort_flag) {
        const uint32_t limit = ch.sync_limit != 0u ? ch.sync_limit : kSyncLimit;
        uint32_t it = 0;
        while (ld_acquire(ch.sync + (p - 1)) < (unsigned)C) {
          if (++it > limit) {
            set_status(status, TQ_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          if (it > 32) __nanosleep(64);
        }
        if (p == 1) grid_dep_launch();
      }
      consumer_sync();
    }
    for (int b = 0; b < a.B; ++b) {
      // -- this CTA's residual rows, read by the epilogues: loaded into
      // registers here and stored to shared memory after the activation loads
      // are issued (one memory round trip for both); the down projection's
      // residual rows are the output projection's outputs of the same CTA
      // (same rows, same tiles), kept in shared memory since phase 0
      const int t0c = u0 / q.G, ntiles = (u1 - u0) / q.G;
      float* rsd = nullptr;
      const bool carried = carry && p == 2;
      const bool keep = carry && p == 0;
      float rv[kResidPerThread];
      if (mode == GEMV_STORE && a.residual != nullptr && a.nseg == 1 && ntiles <= kResidTiles) {
        rsd = reinterpret_cast<float*>(smem + L.resid);
        if (!carried) {
#pragma unroll
          for (int k = 0; k < kResidPerThread; ++k) {
            const int r = tid + k * kCT, row = t0c * kTileRows + r;
            rv[k] = r < ntiles * kTileRows && row < a.N ? __ldcg(a.residual + (int64_t)b * a.N + row) : 0.f;
          }
        }
      }
      // -- activations -> fp16 hi/lo fragments in shared memory.  Pair index
      // (blk, c): inputs 4c..4c+3 and 16+4c..19+4c of block blk; one thread
      // holds up to kPPT pairs in registers across the block reduction.
      const float* xb = a.x + (int64_t)b * a.K;
      const int npairs = a.K / 8;
      float4 v0[kPPT], v1[kPPT];
      float ss = 0.f, mx = 0.f;
#pragma unroll
      for (int r = 0; r < kPPT; ++r) {
        const int pr = tid + r * kCT;
        if (pr < npairs) {
          const int blk = pr >> 2, c = pr & 3;
          v0[r] = __ldcg(reinterpret_cast<const float4*>(xb + blk * 32 + 4 * c));
          v1[r] = __ldcg(reinterpret_cast<const float4*>(xb + blk * 32 + 16 + 4 * c));
          if (a.gain != nullptr) {
            const float4 p0 = v0[r], p1 = v1[r];
            ss = fmaf(p0.x, p0.x, fmaf(p0.y, p0.y, fmaf(p0.z, p0.z, fmaf(p0.w, p0.w, ss))));
            ss = fmaf(p1.x, p1.x, fmaf(p1.y, p1.y, fmaf(p1.z, p1.z, fmaf(p1.w, p1.w, ss))));
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gain + blk * 32 + 4 * c));
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gain + blk * 32 + 16 + 4 * c));
            v0[r] = make_float4(p0.x * g0.x, p0.y * g0.y, p0.z * g0.z, p0.w * g0.w);
            v1[r] = make_float4(p1.x * g1.x, p1.y * g1.y, p1.z * g1.z, p1.w * g1.w);
          }
          mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v0[r].x), fabsf(v0[r].y)), fmaxf(fabsf(v0[r].z), fabsf(v0[r].w))));
          mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v1[r].x), fabsf(v1[r].y)), fmaxf(fabsf(v1[r].z), fabsf(v1[r].w))));
        }
      }
      if (rsd != nullptr && !carried) {
#pragma unroll
        for (int k = 0; k < kResidPerThread; ++k) {
          const int r = tid + k * kCT;
          if (r < ntiles * kTileRows) rsd[r] = rv[k];
        }
      }
      ss = warp_sum(ss);
      mx = warp_max(mx);
      if (lane == 0) {
        sum_sh[warp] = ss;
        max_sh[warp] = mx;
      }
      consumer_sync();
      ss = 0.f;
      mx = 0.f;
      for (int w = 0; w < kW; ++w) {
        ss += sum_sh[w];
        mx = fmaxf(mx, max_sh[w]);
      }
      const float scale = a.gain != nullptr ? 1.0f / sqrtf(ss / (float)a.K + a.eps) : 1.0f;
      mx *= scale;
      int e2 = 0;  // S = 2^e2 puts the largest |value| in [2^14, 2^15)
      if (mx > 0.f && mx <= 3.4e38f) e2 = 14 - (int)((__float_as_uint(mx) >> 23) & 0xffu) + 127;
      e2 = max(-100, min(126, e2));
      const float inv_s = __uint_as_float((uint32_t)(127 - e2) << 23) * 16777216.0f;  // 2^24 / S
      const float f = scale * __uint_as_float((uint32_t)(e2 + 127) << 23);
#pragma unroll
      for (int r = 0; r < kPPT; ++r) {
        const int pr = tid + r * kCT;
        if (pr < npairs) {  // whole warps: npairs is a multiple of 32
          const int blk = pr >> 2, c = pr & 3;
          float e[8] = {v0[r].x * f, v0[r].y * f, v0[r].z * f, v0[r].w * f,
                        v1[r].x * f, v1[r].y * f, v1[r].z * f, v1[r].w * f};
          // code bias x sum of the pair's activations (8 for Q4_0, 128 for Q8_0;
          // AFFINE4: the sum itself, which the group's bias multiplies)
          float bias = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
          bias *= WT == TQ_Q4_0 ? 8.0f : WT == TQ_Q8_0 ? 128.0f : 1.0f;
          if (nib4(WT)) {  // pairs (0,2) (1,3) (4,6)/16 (5,7)/16
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
            const float h0 = __uint_as_float(__float_as_uint(e[2 * k]) & 0xFFFFE000u);  // 11 significant bits
            const float h1 = __uint_as_float(__float_as_uint(e[2 * k + 1]) & 0xFFFFE000u);
            const __half2 hh = __floats2half2_rn(h0, h1);
            const __half2 ll = __floats2half2_rn(e[2 * k] - h0, e[2 * k + 1] - h1);
            hi[k] = *reinterpret_cast<const uint32_t*>(&hh);
            lo[k] = *reinterpret_cast<const uint32_t*>(&ll);
          }
          bias += __shfl_xor_sync(0xffffffffu, bias, 1);
          bias += __shfl_xor_sync(0xffffffffu, bias, 2);
          uint4* slot = reinterpret_cast<uint4*>(smem + L.xtab + blk * kXBlockBytes);
          slot[c] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          slot[4 + c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          if (c == 0) reinterpret_cast<float*>(smem + L.xneg)[blk] = -bias * 5.9604644775390625e-8f;  // 2^-24
        }
      }
      consumer_sync();

      // -- this warp's units
      unsigned long long best = 0ull;
      float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      int cur = -1;
      for (int u = wa; u < wb;) {
        const int t = u / q.G;
        const int n = min(q.k, min((t + 1) * q.G, wb) - u);
        if (t != cur) {
          if (cur >= 0) flush_tile(a, mode, q, b, cur, wa, wb, warp, lane, acc, red, rsd, keep, t0c, inv_s, best);
          cur = t;
          acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
        }
        const int stage = i % depth;
        // Every lane waits.  A timed-out wait sets the status and the abort flag;
        // the loop then runs on without waiting, on stale data, so barriers match.
        const bool ok = *abort_flag != 0 || mbar_wait_bounded(&full[stage], (i / depth) & 1, kWaitLimit);
        if (!__all_sync(0xffffffffu, ok) && lane == 0) {
          set_status(status, TQ_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
        const uint32_t stq = ring_s + stage * F::SLOT;
        const uint32_t std_ = stq + q.mats * q.k * F::QU;
        for (int k = 0; k < n; ++k) {
          const int ub = (u + k - t * q.G) * kUnitBlocks;  // first block of the unit
          const uint32_t xt = xtab + ub * kXBlockBytes, xn = xneg + ub * 4;
          if (mode == GEMV_SWIGLU) {
            unit_dot<WT, 2>(stq + k * F::QU, q.k * F::QU, std_ + k * kUnitD, q.k * kUnitD, xt, xn, lane, acc);
          } else {
            float a1[1][2] = {{acc[0][0], acc[0][1]}};
            unit_dot<WT, 1>(stq + k * F::QU, 0, std_ + k * kUnitD, 0, xt, xn, lane, a1);
            acc[0][0] = a1[0][0];
            acc[0][1] = a1[0][1];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);  // the producer may refill the stage
        u += n;
        ++i;
      }
      if (cur >= 0) flush_tile(a, mode, q, b, cur, wa, wb, warp, lane, acc, red, rsd, keep, t0c, inv_s, best);
      consumer_sync();

      // -- tiles shared between warps (and CTAs): the first contributing warp sums
      if (wa < wb) {
        const int tf = wa / q.G, tl = (wb - 1) / q.G;
        if ((tf * q.G < wa || tf * q.G + q.G > wb) && wa == max(u0, tf * q.G))
          reduce_tile(a, mode, q, b, tf, u0, u1, warp, lane, red, rsd, keep, t0c, inv_s, best);
        if (tl != tf && tl * q.G + q.G > wb)
          reduce_tile(a, mode, q, b, tl, u0, u1, warp, lane, red, rsd, keep, t0c, inv_s, best);
      }

      if (mode == GEMV_ARGMAX) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
          best = other > best ? other : best;
        }
        if (lane == 0) best_sh[warp] = best;
        consumer_sync();
        if (tid == 0) {
          unsigned long long m = 0ull;
          for (int w = 0; w < kW; ++w) m = best_sh[w] > m ? best_sh[w] : m;
          if (m != 0ull) atomicMax(a.argmax_keys + b, m);
        }
      }
      consumer_sync();  // the fragments, partials and sums are rewritten next
    }
    // this CTA's outputs of phase p are complete: tell the other CTAs
    if (p + 1 < ch.n && tid == 0) {
      __threadfence();
      atomicAdd(ch.sync + p, 1u);
    }
  }
  // the last CTA out resets the counters for the next launch
  if (ch.n > 1 && tid == 0) {
    if (atomicAdd(ch.sync + kMaxPhases, 1u) == (unsigned)C - 1) {
      for (int p = 0; p <= kMaxPhases; ++p) ch.sync[p] = 0u;
      __threadfence();
    }
  }
}

// Ring depth from the shared-memory budget; grid = one CTA per SM (fewer for
// a single small GEMV).
template <int WT>
cudaError_t launch_chain(const GemvChain& c, cudaStream_t s) {
  using F = Fmt<WT>;
  static PerDevice setup;
  int sms = 0;
  cudaError_t e = per_device(setup, &sms, [](int dev, int& n) {
    cudaError_t r = cudaFuncSetAttribute(gemv_chain_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemMax);
    if (r != cudaSuccess) return r;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kNumSMs;
    if (n > kMaxGrid) n = kMaxGrid;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  int max_k = 0;
  for (int p = 0; p < c.n; ++p) max_k = c.ph[p].K > max_k ? c.ph[p].K : max_k;
  int depth = 8;
  while (depth > 1 && smem_layout(F::SLOT, depth, max_k).bytes > kSmemMax) --depth;
  const Smem L = smem_layout(F::SLOT, depth, max_k);
  if (L.bytes > kSmemMax) return cudaErrorInvalidValue;
  if (c.n == 1) {
    const Geo q = geo_of(c.ph[0], c.mode[0], sms, F::SU);
    return launch_k(gemv_chain_kernel<WT>, dim3(q.Cp), dim3(kThreads), L.bytes, s, c, depth, max_k);
  }
  // several phases: every CTA must be resident at once (grid-wide counters).
  // The grid is one CTA per SM (a CTA fits an SM), the CTAs start as the
  // previous kernel's CTAs exit, and the kernel releases its dependent launch
  // only when all of them are running.
  // Without programmatic dependent launch (TQ_PDL=0) a cooperative launch.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L.bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_chain_kernel<WT>, c, depth, max_k);
}

}  // namespace gemv
}  // namespace tq
