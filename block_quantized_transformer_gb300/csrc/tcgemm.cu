// Tensor-core (tcgen05 / TMEM) GEMM over the tiled Q4_0 / Q8_0 weights, for
// the projections of prefill and of batched decode, where many token rows
// share each weight: Y[t][r] = sum_k W[r][k] X[t][k] (+ residual).  The
// prompt pass of "Всередині LLM: чисте виконання на Python для Qwen3-0.6B на
// MLX" (steps 3-7 over all positions, step 9: prefill, then one token at a
// time) is the same set of dense contractions over T rows.
//
// Operands.  The weights are decoded to fp16 in shared memory, one rounding
// of the exact product d * (q - 8) (Q4_0) or d * q (Q8_0); the activation
// rows are turned into fp16 after a power-of-two scale per row (xprep16),
// so that the row's largest magnitude lies in [2^14, 2^15); the tensor core
// multiplies fp16 x fp16 and sums in f32 (TMEM), and the epilogue undoes the
// row scale exactly.  Each operand is rounded once to 11 significant bits,
// so an output differs from the exact sum by at most about 2^-10 * sum|x w|.
//
// CTA work item: 128 weight rows (8 tiles of 16) x BN token rows over a
// range of K units (the whole K, or a 1/ks share when few CTAs would be busy:
// the ks partial sums are then added by the last CTA of the group, in split
// order).  K advances in stages of 128 inputs.  Roles:
//  - warp 18, lane 0: streams the CTA's weight units (codes and scales of
//    its 8 tiles, runs of U units of 256 inputs) into a ring of R
//    shared-memory slots with 1-D bulk copies (TMA engine); weights are
//    read-only, so this starts before the preceding kernel is done;
//  - 16 decode warps: warp w owns TMEM lanes 32 (w % 4) .. + 31 (one weight
//    row per thread) and one code word of each of the stage's 4 blocks; it
//    decodes its 32 weights from the raw slot to fp16 and writes them with
//    tcgen05.st into one of NA weight-operand stages held in tensor memory
//    (64 columns each), so the decoded weights never pass through shared
//    memory, whose bandwidth the tensor core's reads of the activations need;
//  - warp 16: allocates the CTA's 512 TMEM columns (NI accumulators of BN
//    columns, then the weight stages), and its lane 0 loads each stage's
//    activations with two TMA tile loads (64 inputs x BN rows, 128-byte
//    swizzle) from the fp16 activation matrix into one of NB shared stages;
//  - warp 17 (and warp 19 when NI = 2), lane 0: issues a stage's 8
//    tcgen05.mma (M 128, N BN, K 16; A from TMEM, B from shared memory) into
//    its own accumulator, the two taking alternate stages, and commits them
//    to the stages' "empty" barriers, after its last stage to the
//    accumulator barrier.  An MMA of few columns costs the issuing thread
//    about as much as one of many (measured: ~60 cycles at N 32, plus
//    ~500 cycles of barrier waits and commits per stage), so at N <= 128 one
//    issuer would pace the whole CTA;
//  - epilogue (decode warps 0-7, or 0-3 for 32 columns; 32 TMEM lanes
//    each): TMEM -> registers (the NI accumulators summed in order), times
//    the row scale, plus the residual (all loads of a chunk before its
//    stores), to global memory.
// Every wait is bounded in time; a wait that gives up sets
// TQ_DEV_WAIT_TIMEOUT and the CTA runs on without waiting, then waits
// (bounded) for its MMAs and copies before it frees TMEM and exits.
#include <type_traits>

#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"
#include "tmap.cuh"
#include "umma.cuh"

namespace tq {
namespace tc {

constexpr int kBM = 128;          // weight rows per CTA
constexpr int kBK = 128;          // inputs per operand stage (half a unit; two swizzle atoms of activations)
constexpr int kTiles = kBM / kTileRows;
constexpr int kDQ = 16;           // decode warps, warp w <-> rows 8 (w % 2) .. of tile w / 2
constexpr int kWarpB = kDQ, kWarpMMA = kDQ + 1, kWarpRaw = kDQ + 2, kWarpMMA2 = kDQ + 3;
constexpr int kThreads = (kDQ + 4) * 32;
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s: far beyond any legitimate wait here
constexpr int kSmemBudget = 212 * 1024;

template <int WT, int BN>
struct Cfg {
  // Rings: weight operands in TMEM (NA stages of 64 columns after the BN
  // accumulator columns), activation operands in shared memory (NB stages of
  // 128 inputs x BN rows), raw weight units in shared memory (R slots of 256
  // inputs x 128 rows).  A stage returns to its producer only after the MMAs
  // that read it complete, so each ring covers its own round trip.
  static constexpr uint32_t TMEM_COLS = 512;
  // MMA issuers: one tcgen05.mma with few columns costs its issuing thread
  // about as much as one with many, so up to 128 columns two threads issue
  // alternate stages, each into its own accumulator (summed in the epilogue)
  static constexpr int NI = BN <= 128 ? 2 : 1;
  static constexpr int ACC = NI * BN;  // accumulator columns
  static constexpr int NA0 = (int)(TMEM_COLS - ACC) / 64;
  static constexpr int NA = NA0 > 6 ? 6 : NA0;
  static constexpr int B = BN * kBK * 2;                       // BN * 256 bytes
  static constexpr int NB0 = (BN >= 256 ? 128 * 1024 : 64 * 1024) / B;
  static constexpr int NB = NB0 < 2 ? 2 : NB0 > 8 ? 8 : NB0;
  static constexpr int UQ = unit_qs_bytes(WT);                 // codes of one tile's unit
  static constexpr int RAW1 = kTiles * (UQ + kUnitD);          // the CTA's 8 tiles, one unit each
  // a raw slot holds U consecutive units of every tile, so each tile's run
  // arrives in two bulk copies (codes, scales) of several KB: the TMA
  // engine's cost per copy stays small against its cost per byte
  static constexpr int U0 = (kSmemBudget - NB * B) / (2 * RAW1);
  static constexpr int U = U0 >= 4 ? 4 : U0 >= 2 ? 2 : 1;
  static constexpr int RAW = U * RAW1;
  static constexpr int R0 = (kSmemBudget - NB * B) / RAW;
  static constexpr int R = R0 > 4 ? 4 : R0;                    // raw slots
  static constexpr int MISC = 512;                             // barriers, TMEM address, flags
  static constexpr int SMEM = 1024 + NB * B + R * RAW + MISC;  // + alignment slack
  static_assert(NA >= 3, "tensor memory too small for the weight stages");
  static_assert(R >= 2, "shared memory too small for two raw slots");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct TileMap {
  int T;
  int tile0[4];
  int row0[3];
};

__host__ __device__ inline TileMap tile_map(const TcGemmArgs& a) {
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

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             uint32_t* status) {
  if (*abort_flag) return false;
  if (mbar_wait_timed(bar, parity, kWaitNs)) return true;
  set_status(status, TQ_DEV_WAIT_TIMEOUT);
  *abort_flag = 1;
  return false;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Four codes held as the bytes of `w` -> fp16 (code - bias) * d, as two
// pairs: each byte b is interleaved with 0x64, which reads as the fp16 value
// 1024 + b; subtracting bias (1024 + the code offset) is exact, and the
// product with the block scale is the one rounding.
__device__ __forceinline__ void decode4(uint32_t w, __half2 bias2, __half2 d2, uint32_t& p01, uint32_t& p23) {
  const uint32_t a = __byte_perm(w, 0x64646464u, 0x5150);  // fp16 pair 1024 + byte0, 1024 + byte1
  const uint32_t b = __byte_perm(w, 0x64646464u, 0x5352);  // bytes 2, 3
  p01 = h2bits(__hmul2(__hsub2(*reinterpret_cast<const __half2*>(&a), bias2), d2));
  p23 = h2bits(__hmul2(__hsub2(*reinterpret_cast<const __half2*>(&b), bias2), d2));
}

// AFFINE4: four codes -> fp16 q s + b (q = (1024 + q) - 1024 exactly, then
// one fused multiply-add).
__device__ __forceinline__ void decode4_affine(uint32_t w, __half2 off2, __half2 s2, __half2 b2, uint32_t& p01,
                                               uint32_t& p23) {
  const uint32_t a = __byte_perm(w, 0x64646464u, 0x5150);
  const uint32_t b = __byte_perm(w, 0x64646464u, 0x5352);
  p01 = h2bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&a), off2), s2, b2));
  p23 = h2bits(__hfma2(__hsub2(*reinterpret_cast<const __half2*>(&b), off2), s2, b2));
}

__device__ __forceinline__ __half2 scale2(uint32_t bits) {
  const __half h = __ushort_as_half((uint16_t)(bits & 0xffffu));
  return __halves2half2(h, h);
}

// Inputs inside each 128-input half unit are taken in the order the tiled
// layout hands them to a thread: position p = 32 i + 8 jb + e (word i,
// block jb, e < 8) holds input 32 jb + 4 i + (e & 3) + 16 (e >> 2), i.e.
// word i's four low-nibble (or first) inputs, then its four high-nibble (or
// second-word) inputs.  xprep16 writes the activations in the same order,
// so the contraction is unchanged.
//
// Per-thread constants of the decode.  Decode warp w owns TMEM lanes
// 32 (w % 4) .. + 31, so lane l holds weight row r = 32 (w % 4) + l (tile
// r / 16, row r % 16 = 8 h + g of the tile), and decodes code word i = w / 4
// of each of the stage's 4 blocks: 32 inputs, TMEM columns 16 i .. 16 i + 15
// of the stage.
struct DecodeLane {
  uint32_t qs;      // raw-slot offset of the thread's code piece (first unit, stage 0)
  uint32_t dd;      // raw-slot offset of the row's scales of blocks 0..3 (first unit)
  uint32_t col;     // TMEM lane << 16 | column offset within a stage
  bool ok;          // the tile exists
};

template <int WT, int U>
__device__ __forceinline__ DecodeLane decode_lane(int lane, int w, bool tile_ok) {
  constexpr int UQ = unit_qs_bytes(WT);
  const int q = w & 3, i = w >> 2;
  const int r = 32 * q + lane, tw = r >> 4, rr = r & 15, h = rr >> 3, g = rr & 7;
  DecodeLane d;
  // Q4_0: the 16-byte piece (h*2 + j/4)*32 + 4g + i holds word i of blocks 4(j/4) .. +3;
  // Q8_0: the piece (h*4 + j/2)*32 + 4g + i holds code words i, i + 4 of blocks 2(j/2), +1
  d.qs = (uint32_t)(tw * U * UQ + ((nib4(WT) ? h * 2 : h * 4) * 32 + 4 * g + i) * 16);
  d.dd = (uint32_t)(kTiles * U * UQ + tw * U * kUnitD + (h * 8 + g) * 16);
  d.col = ((uint32_t)(32 * q) << 16) | (uint32_t)(16 * i);
  d.ok = tile_ok;
  return d;
}

// Stage S of a unit (inputs 128 S .. 128 S + 127: blocks 4S .. 4S + 3) ->
// this thread's 32 fp16 weights as 16 TMEM columns.  rq, rd: the unit's
// codes and scales in the raw slot (which holds the 8 tiles' runs of U units
// of codes, UQ bytes each, then their scales, 256 B each).
template <int WT, int S>
__device__ __forceinline__ void decode_stage(uint32_t rq, uint32_t rd, const DecodeLane& L, uint32_t (&out)[16]) {
  if (!L.ok) {  // rows past the last tile: zeros
#pragma unroll
    for (int k = 0; k < 16; ++k) out[k] = 0u;
    return;
  }
  const uint2 dv = lds64(rd + L.dd + 8 * S);  // scales of blocks 4S .. 4S + 3 (AFFINE4: s, b of 2 groups)
  const uint32_t ds[2] = {dv.x, dv.y};
  const __half2 bias2 = __float2half2_rn(WT == TQ_Q4_0 ? 1032.f : WT == TQ_Q8_0 ? 1152.f : 1024.f);
  uint32_t lo[4], hi[4];  // per block: first and second four inputs of word i
  if (nib4(WT)) {
    const uint4 v = lds128(rq + L.qs + S * 512);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) {
      lo[jb] = wv[jb] & 0x0F0F0F0Fu;
      hi[jb] = (wv[jb] >> 4) & 0x0F0F0F0Fu;
    }
  } else {
#pragma unroll
    for (int jp = 0; jp < 2; ++jp) {
      const uint4 v = lds128(rq + L.qs + (2 * S + jp) * 512);
      lo[2 * jp] = v.x ^ 0x80808080u;
      hi[2 * jp] = v.y ^ 0x80808080u;
      lo[2 * jp + 1] = v.z ^ 0x80808080u;
      hi[2 * jp + 1] = v.w ^ 0x80808080u;
    }
  }
  if (WT == TQ_AFFINE4) {
    // group of blocks (2k, 2k+1): bf16 scale and bias in element pair k,
    // converted to fp16 (exact within fp16's range); one fused rounding of q s + b
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const __half2 s2 = __float2half2_rn(__uint_as_float(ds[k] << 16));
      const __half2 b2 = __float2half2_rn(__uint_as_float(ds[k] & 0xffff0000u));
#pragma unroll
      for (int jb = 2 * k; jb < 2 * k + 2; ++jb) {
        decode4_affine(lo[jb], bias2, s2, b2, out[4 * jb], out[4 * jb + 1]);
        decode4_affine(hi[jb], bias2, s2, b2, out[4 * jb + 2], out[4 * jb + 3]);
      }
    }
  } else {
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) {
      const __half2 d2 = scale2(ds[jb >> 1] >> (16 * (jb & 1)));
      decode4(lo[jb], bias2, d2, out[4 * jb], out[4 * jb + 1]);
      decode4(hi[jb], bias2, d2, out[4 * jb + 2], out[4 * jb + 3]);
    }
  }
}

template <int WT, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tcgemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ TcGemmArgs a) {
  using C = Cfg<WT, BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw0 = smem_addr(smem_raw);
  const uint32_t base = (raw0 + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw0);
  const uint32_t bbase = base;                                  // activation stages
  const uint32_t rbase = bbase + C::NB * C::B;                  // raw slots
  uint8_t* misc = sbase + (rbase - base) + C::R * C::RAW;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);          // [NA] weight operand in TMEM
  uint64_t* empty = full + C::NA;                               // [NA] weight operand consumed
  uint64_t* bfull = empty + C::NA;                              // [NB] activation operand landed
  uint64_t* bempty = bfull + C::NB;                             // [NB] activation operand consumed
  uint64_t* rfull = bempty + C::NB;                             // [R] raw slot landed
  uint64_t* rempty = rfull + C::R;                              // [R] raw slot decoded
  uint64_t* acc_bar = rempty + C::R;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* last_flag = abort_flag + 1;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const TileMap m = tile_map(a);
  const int G = a.K / 256;
  const int ks = gridDim.z, z = blockIdx.z;
  const int ub = G * z / ks, ue = G * (z + 1) / ks;  // this CTA's K units
  const int nu = ue - ub, nst = 2 * nu;
  const int tile = blockIdx.x * kTiles;
  const int n0 = blockIdx.y * BN;

  if (tid == 0) {
    for (int k = 0; k < C::NA; ++k) {
      mbar_init(&full[k], kDQ);
      mbar_init(&empty[k], 1);
    }
    for (int k = 0; k < C::NB; ++k) {
      mbar_init(&bfull[k], 1);
      mbar_init(&bempty[k], 1);
    }
    for (int k = 0; k < C::R; ++k) {
      mbar_init(&rfull[k], 1);
      mbar_init(&rempty[k], kDQ);
    }
    mbar_init(acc_bar, C::NI);
    *abort_flag = 0;
    fence_proxy_async();
  }
  if (warp == kWarpB) umma::tmem_alloc(tmem_holder, C::TMEM_COLS);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  grid_dep_launch();

  if (warp < kDQ) {
    // ------------------------------------------------------------ decode
    const DecodeLane L = decode_lane<WT, C::U>(lane, warp, tile + ((32 * (warp & 3) + lane) >> 4) < m.T);
    auto stage = [&](auto qc, int u, uint32_t rq, uint32_t rd) {
      constexpr int S = decltype(qc)::value;
      const int s = 2 * u + S, slot = s % C::NA;
      uint32_t w32[16];
      decode_stage<WT, S>(rq, rd, L, w32);
      if (s >= C::NA) wait_bounded(&empty[slot], (uint32_t)(((s / C::NA) - 1) & 1), abort_flag, a.status);
      umma::fence_after_sync();
      umma::tmem_st16(tmem + L.col + (uint32_t)(C::ACC + 64 * slot), w32);
      umma::fence_before_sync();  // the stores, before the MMA thread learns of them
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[slot]);
    };
    const int nslots = (nu + C::U - 1) / C::U;
    for (int k = 0; k < nslots; ++k) {
      const int rsl = k % C::R;
      wait_bounded(&rfull[rsl], (uint32_t)((k / C::R) & 1), abort_flag, a.status);
      const uint32_t rs = rbase + rsl * C::RAW;
      const int n = min(C::U, nu - k * C::U);
      for (int uu = 0; uu < n; ++uu) {
        const uint32_t rq = rs + uu * C::UQ, rd = rs + uu * kUnitD;
        stage(std::integral_constant<int, 0>{}, k * C::U + uu, rq, rd);
        stage(std::integral_constant<int, 1>{}, k * C::U + uu, rq, rd);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[rsl]);
    }
    // ---------------------------------------------------------- epilogue
    constexpr int EW = BN >= 64 ? 8 : 4;        // epilogue warps
    constexpr int CW = BN >= 64 ? BN / 2 : BN;  // columns per epilogue warp
    if (warp < EW) {
      grid_dep_wait();
      wait_bounded(acc_bar, 0u, abort_flag, a.status);
      umma::fence_after_sync();
      const int qd = warp & 3;                // TMEM lanes 32 qd .. 32 qd + 31
      const int row = 32 * qd + lane;         // weight row within the CTA
      const int t = tile + row / kTileRows;
      const bool row_ok = t < m.T;
      const int sg = row_ok ? seg_of(m, t) : 0;
      const int local = row_ok ? (t - m.tile0[sg]) * kTileRows + row % kTileRows : 0;
      const bool valid = row_ok && local < a.seg[sg].rows;
      const int col = (sg == 0 ? m.row0[0] : sg == 1 ? m.row0[1] : m.row0[2]) + local;
      const float bcol = valid && a.bias != nullptr && ks == 1 ? __ldg(a.bias + col) : 0.f;
      const int c0 = (warp >> 2) * CW;
      for (int cc = 0; cc < CW; cc += 16) {
        float v[16];
        umma::tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(c0 + cc), v);
        if (C::NI > 1) {  // the second issuer's accumulator (odd stages; every CTA has at least two stages)
          float v2[16];
          umma::tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(BN + c0 + cc), v2);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += v2[j];
        }
        if (!valid) continue;
        const int tk0 = n0 + c0 + cc;
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= tk0 + j < a.T ? __ldg(a.inv_s + tk0 + j) : 0.f;
        if (ks > 1) {
          float* dst = a.part + (int64_t)z * a.T * a.ldy + col;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (tk0 + j < a.T) __stcg(dst + (int64_t)(tk0 + j) * a.ldy, v[j]);
        } else if (a.residual != nullptr) {
          // every residual load before any store (the residual may alias y)
          float r[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            r[j] = tk0 + j < a.T ? __ldcg(a.residual + (int64_t)(tk0 + j) * a.ldy + col) : 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (tk0 + j < a.T) a.y[(int64_t)(tk0 + j) * a.ldy + col] = (r[j] + v[j]) + bcol;
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (tk0 + j < a.T) a.y[(int64_t)(tk0 + j) * a.ldy + col] = v[j] + bcol;
        }
      }
    }
  } else if (warp == kWarpB) {
    // ------------------------------------------------- activations (TMA)
    if (lane == 0) {
      umma::prefetch_tmap(&xmap);
      grid_dep_wait();
      int issued = 0;
      for (int s = 0; s < nst; ++s) {
        const int slot = s % C::NB;
        if (s >= C::NB && !wait_bounded(&bempty[slot], (uint32_t)(((s / C::NB) - 1) & 1), abort_flag, a.status))
          break;
        if (*abort_flag) break;
        mbar_arrive_expect_tx(&bfull[slot], (uint32_t)C::B);
        uint8_t* dst = sbase + (bbase - base) + slot * C::B;
        const int k0 = (2 * ub + s) * kBK;
        umma::tma_load_2d(dst, &xmap, k0, n0, &bfull[slot]);
        umma::tma_load_2d(dst + BN * 128, &xmap, k0 + 64, n0, &bfull[slot]);
        ++issued;
      }
      // every issued load lands before the CTA's shared memory is released
      for (int s = (issued > C::NB ? issued - C::NB : 0); s < issued; ++s)
        mbar_wait_timed(&bfull[s % C::NB], (uint32_t)((s / C::NB) & 1), kWaitNs);
    }
  } else if (warp == kWarpMMA || (C::NI > 1 && warp == kWarpMMA2)) {
    // ------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = umma::idesc_f16_f32(kBM, BN);
      const int par = warp == kWarpMMA ? 0 : 1;  // stages par, par + NI, ...
      const uint32_t D = tmem + (uint32_t)(par * BN);
      for (int s = par; s < nst; s += C::NI) {
        const int slot = s % C::NA, bslot = s % C::NB;
        const bool ok = wait_bounded(&full[slot], (uint32_t)((s / C::NA) & 1), abort_flag, a.status) &&
                        wait_bounded(&bfull[bslot], (uint32_t)((s / C::NB) & 1), abort_flag, a.status);
        umma::fence_after_sync();
        const uint32_t A = tmem + (uint32_t)(C::ACC + 64 * slot), B = bbase + bslot * C::B;
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_f16_tmem_a(D, A + 8 * kk, umma::desc_sw128(B + (kk >> 2) * (BN * 128) + (kk & 3) * 32),
                                 idesc, (s > par || kk > 0) ? 1u : 0u);
        }
        umma::commit(&empty[slot]);  // both stages are free once these MMAs are done
        umma::commit(&bempty[bslot]);
      }
      umma::commit(acc_bar);
    }
  } else if (warp == kWarpRaw) {
    // ------------------------------------------------- weight units (bulk)
    if (lane == 0) {
      int nt = 0;  // the CTA's tiles that exist
      for (int i = 0; i < kTiles; ++i)
        if (tile + i < m.T) ++nt;
      const int nslots = (nu + C::U - 1) / C::U;
      int issued = 0;
      for (int k = 0; k < nslots; ++k) {
        const int rsl = k % C::R;
        if (k >= C::R && !wait_bounded(&rempty[rsl], (uint32_t)(((k / C::R) - 1) & 1), abort_flag, a.status))
          break;
        if (*abort_flag) break;
        const int n = min(C::U, nu - k * C::U);  // units in this slot
        uint8_t* dst = sbase + (rbase - base) + rsl * C::RAW;
        mbar_arrive_expect_tx(&rfull[rsl], (uint32_t)(nt * n * (C::UQ + kUnitD)));
        for (int i = 0; i < nt; ++i) {
          const int t = tile + i, sg = seg_of(m, t);
          const GemvSeg& gs = a.seg[sg];
          const int64_t unit = (int64_t)(t - m.tile0[sg]) * G + ub + k * C::U;  // a tile's units are contiguous
          bulk_g2s(dst + i * C::U * C::UQ, gs.qs + unit * C::UQ, (uint32_t)(n * C::UQ), &rfull[rsl]);
          bulk_g2s(dst + kTiles * C::U * C::UQ + i * C::U * kUnitD,
                   reinterpret_cast<const uint8_t*>(gs.d) + unit * kUnitD, (uint32_t)(n * kUnitD), &rfull[rsl]);
        }
        ++issued;
      }
      // every issued copy lands before the CTA's shared memory is released
      for (int k = (issued > C::R ? issued - C::R : 0); k < issued; ++k)
        mbar_wait_timed(&rfull[k % C::R], (uint32_t)((k / C::R) & 1), kWaitNs);
    }
  }

  if (ks > 1) __threadfence();  // this thread's partial sums, before the split counter
  // every TMEM load and every MMA is done before the columns are freed
  umma::fence_before_sync();
  __syncthreads();
  if (warp == kWarpB) {
    umma::fence_after_sync();
    if (*abort_flag) mbar_wait_timed(acc_bar, 0u, kWaitNs);
    umma::tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (ks == 1) return;

  // ---------------------------------------------- split K: the last CTA adds
  if (tid == 0) {
    __threadfence();
    unsigned* ctr = a.counters + blockIdx.y * gridDim.x + blockIdx.x;
    const int last = atomicAdd(ctr, 1u) == (unsigned)(ks - 1);
    if (last) {
      *ctr = 0u;  // zero for the next launch
      __threadfence();
    }
    *last_flag = last;
  }
  __syncthreads();
  if (!*last_flag) return;
  // Groups of 4 consecutive rows of one token -> threads.  Every partial sum
  // of a group (8 splits at a time) and its residual are loaded before any
  // add, as float4 where the group is whole and 16-byte aligned; the adds
  // run in split order.
  const bool vec = (a.ldy & 3) == 0 && (m.row0[1] & 3) == 0 && (m.row0[2] & 3) == 0 &&
                   ((reinterpret_cast<uintptr_t>(a.y) | reinterpret_cast<uintptr_t>(a.part) |
                     reinterpret_cast<uintptr_t>(a.residual) | reinterpret_cast<uintptr_t>(a.bias)) & 15u) == 0;
  const int64_t pstride = (int64_t)a.T * a.ldy;
  for (int gi = tid; gi < (kBM / 4) * BN; gi += kThreads) {
    const int row = 4 * (gi % (kBM / 4)), tok = n0 + gi / (kBM / 4);
    const int t = tile + row / kTileRows;
    if (t >= m.T || tok >= a.T) continue;
    const int sg = seg_of(m, t);
    const int local = (t - m.tile0[sg]) * kTileRows + row % kTileRows;
    const int rows = a.seg[sg].rows;
    if (local >= rows) continue;
    const int col = (sg == 0 ? m.row0[0] : sg == 1 ? m.row0[1] : m.row0[2]) + local;
    const int64_t off = (int64_t)tok * a.ldy + col;
    if (vec && local + 4 <= rows) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 r = a.residual != nullptr ? __ldcg(reinterpret_cast<const float4*>(a.residual + off)) : v;
      for (int z0 = 0; z0 < ks; z0 += 8) {
        float4 p[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (z0 + j < ks) p[j] = __ldcg(reinterpret_cast<const float4*>(a.part + (int64_t)(z0 + j) * pstride + off));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (z0 + j < ks) {  // split order
            v.x += p[j].x;
            v.y += p[j].y;
            v.z += p[j].z;
            v.w += p[j].w;
          }
      }
      const float4 b = a.bias != nullptr ? __ldg(reinterpret_cast<const float4*>(a.bias + col))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(a.y + off) =
          make_float4((r.x + v.x) + b.x, (r.y + v.y) + b.y, (r.z + v.z) + b.z, (r.w + v.w) + b.w);
    } else {
      const int n = min(4, rows - local);
      for (int k = 0; k < n; ++k) {
        float v = 0.f;
        const float r = a.residual != nullptr ? __ldcg(a.residual + off + k) : 0.f;
        for (int zz = 0; zz < ks; ++zz) v += __ldcg(a.part + (int64_t)zz * pstride + off + k);  // split order
        a.y[off + k] = (r + v) + (a.bias != nullptr ? __ldg(a.bias + col + k) : 0.f);
      }
    }
  }
}

// ------------------------------------------------------------ xprep16 --

// Row t of the phase input (x, RMS-normalised with `gain`, or act(x) * up)
// -> fp16 row t of x16 after the power-of-two scale 2^e that puts its largest
// magnitude in [2^14, 2^15), inputs in the word-major order of the GEMM's
// weight operand; inv_s[t] = 2^-e.
__global__ void __launch_bounds__(256) xprep16_kernel(const XPrep16Args a) {
  grid_dep_launch();
  grid_dep_wait();
  constexpr int CPT = 12288 / 8 / 256;  // 8-input chunks per thread at the largest K
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float sum_sh[8], max_sh[8];
  const int nch = a.K / 8;
  const float* xr = a.x + (int64_t)t * a.ldx;
  const float* ur = a.up != nullptr ? a.up + (int64_t)t * a.ldx : nullptr;
  float4 v0[CPT], v1[CPT];
  float ss = 0.f, mx = 0.f;
#pragma unroll
  for (int r = 0; r < CPT; ++r) {
    const int c = tid + r * 256;
    if (c < nch) {
      // output chunk c = positions 8c .. 8c + 7 of the word-major order: word
      // i, block jb of its 128-input half unit
      const int in0 = (c >> 4) * 128 + 32 * (c & 3) + 4 * ((c >> 2) & 3), in1 = in0 + 16;
      float4 p0 = *reinterpret_cast<const float4*>(xr + in0);
      float4 p1 = *reinterpret_cast<const float4*>(xr + in1);
      if (ur != nullptr) {  // act(gate) * up
        const float4 u0 = *reinterpret_cast<const float4*>(ur + in0);
        const float4 u1 = *reinterpret_cast<const float4*>(ur + in1);
        p0 = make_float4(gate_act(p0.x, a.act) * u0.x, gate_act(p0.y, a.act) * u0.y, gate_act(p0.z, a.act) * u0.z,
                         gate_act(p0.w, a.act) * u0.w);
        p1 = make_float4(gate_act(p1.x, a.act) * u1.x, gate_act(p1.y, a.act) * u1.y, gate_act(p1.z, a.act) * u1.z,
                         gate_act(p1.w, a.act) * u1.w);
      }
      if (a.gain != nullptr) {
        ss = fmaf(p0.x, p0.x, fmaf(p0.y, p0.y, fmaf(p0.z, p0.z, fmaf(p0.w, p0.w, ss))));
        ss = fmaf(p1.x, p1.x, fmaf(p1.y, p1.y, fmaf(p1.z, p1.z, fmaf(p1.w, p1.w, ss))));
        const float4 g0 = *reinterpret_cast<const float4*>(a.gain + in0);
        const float4 g1 = *reinterpret_cast<const float4*>(a.gain + in1);
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
  int e2 = 0;  // 2^e2 puts the largest |value| in [2^14, 2^15)
  if (mx > 0.f && mx <= 3.4e38f) e2 = 14 - (int)((__float_as_uint(mx) >> 23) & 0xffu) + 127;
  e2 = max(-100, min(100, e2));
  const float f = scale * __uint_as_float((uint32_t)(e2 + 127) << 23);
  if (tid == 0) a.inv_s[t] = __uint_as_float((uint32_t)(127 - e2) << 23);
  __half* out = a.x16 + (int64_t)t * a.K;
#pragma unroll
  for (int r = 0; r < CPT; ++r) {
    const int c = tid + r * 256;
    if (c < nch) {
      const __half2 h0 = __floats2half2_rn(v0[r].x * f, v0[r].y * f);
      const __half2 h1 = __floats2half2_rn(v0[r].z * f, v0[r].w * f);
      const __half2 h2 = __floats2half2_rn(v1[r].x * f, v1[r].y * f);
      const __half2 h3 = __floats2half2_rn(v1[r].z * f, v1[r].w * f);
      *reinterpret_cast<uint4*>(out + 8 * c) = make_uint4(h2bits(h0), h2bits(h1), h2bits(h2), h2bits(h3));
    }
  }
}

// ------------------------------------------------------------ launch --

// Tensor map of the fp16 activations [T][K]: boxes of 64 inputs x BN rows,
// 128-byte swizzle; rows past T read as zeros.
cudaError_t encode_x(CUtensorMap* map, const __half* x16, int K, int T, int BN) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)BN};
  return tmap_f16_sw128(map, x16, 2, dims, strides, box);
}

template <int WT, int BN>
cudaError_t launch_bn(const TcGemmArgs& a, cudaStream_t s) {
  using C = Cfg<WT, BN>;
  static PerDevice setup;
  int sms = 0;
  cudaError_t e = per_device(setup, &sms, [](int dev, int& n) {
    cudaError_t r = cudaFuncSetAttribute(tcgemm_kernel<WT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (r != cudaSuccess) return r;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kNumSMs;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  CUtensorMap map;
  if ((e = encode_x(&map, a.x16, a.K, a.T, BN)) != cudaSuccess) return e;
  const TileMap m = tile_map(a);
  dim3 grid((m.T + kTiles - 1) / kTiles, (a.T + BN - 1) / BN, 1);
  // Few CTAs, or a last wave that leaves most SMs idle: split K so that
  // waves x (units per split + about one unit of pipeline fill), plus a small
  // cost per split for the partial sums, is least.
  const int G = a.K / 256, base = (int)(grid.x * grid.y);
  if (a.part != nullptr && a.counters != nullptr && base <= a.n_counters) {
    double best = 1e30;
    for (int k = 1; k <= 16 && k <= G; ++k) {
      if (k > 1 && (int64_t)k * a.T * a.ldy > a.part_cap) break;
      const double cost =
          (double)((base * k + sms - 1) / sms) * ((G + k - 1) / k + 1) + (k > 1 ? 0.25 * k : 0.0);
      if (cost < best) {
        best = cost;
        grid.z = k;
      }
    }
  }
  return launch_k(tcgemm_kernel<WT, BN>, grid, dim3(kThreads), C::SMEM, s, map, a);
}

template <int WT>
cudaError_t launch_wt(const TcGemmArgs& a, cudaStream_t s) {
  if (a.T <= 32) return launch_bn<WT, 32>(a, s);
  if (a.T <= 64) return launch_bn<WT, 64>(a, s);
  if (a.T <= 128) return launch_bn<WT, 128>(a, s);
  return launch_bn<WT, 256>(a, s);
}

}  // namespace tc

cudaError_t launch_xprep16(const XPrep16Args& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.K % 256 != 0 || a.K > 12288) return cudaErrorInvalidValue;
  return launch_k(tc::xprep16_kernel, dim3(a.T), dim3(256), 0, s, a);
}

cudaError_t launch_tcgemm(int wtype, const TcGemmArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.K % 256 != 0 || a.K > 12288 || a.nseg < 1 || a.nseg > 3) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.x16) & 15u) != 0) return cudaErrorInvalidValue;
  if (wtype == TQ_AFFINE4) return tc::launch_wt<TQ_AFFINE4>(a, s);
  return wtype == TQ_Q4_0 ? tc::launch_wt<TQ_Q4_0>(a, s) : tc::launch_wt<TQ_Q8_0>(a, s);
}

}  // namespace tq
