// Prefill attention over an f16 cache: every prompt row attends to its causal
// prefix (also the prompt chunks inside a continuous-batching step) ("Всередині LLM: чисте виконання на Python для Qwen3-0.6B на MLX",
// step 5, "Вся функція уваги": softmax(q k^T / sqrt(hd)) v with the causal
// mask over the whole prompt; query head h reads KV head h / G).  The rows
// were normalised, rotated and appended to the cache by rope_append.
//
// Flash-attention layout: one CTA per (block of query tokens, KV head) takes
// 128 query rows, the BQ = 128 / G tokens of the block times the G query
// heads that share the KV head (row r: token r / G, head r % G); 8 warps of
// 16 rows each.  The block's causal key range goes through shared memory in
// tiles of 64 keys, each staged by the TMA engine as 128-byte swizzled boxes
// of 32 keys x 64 dimensions (tensor maps over this layer's K and V caches;
// boxes past the cache's end read as zeros), in a ring of NS stages filled by
// one producer warp.  Per tile and warp, on mma.m16n8k16 with f32 sums:
//  * S = Q K^T: Q as an unevaluated sum hi + lo of two fp16 values after a
//    power-of-two scale per row (21 significant bits), K exact (the cache is
//    f16) read with ldmatrix;
//  * online base-2 softmax on the score fragments, keys past a row's position
//    masked;
//  * O += P V: the probabilities in fp16 (one rounding), V exact, read with
//    ldmatrix.trans.
// A warp skips the tiles past its last row's position.  Every wait is bounded
// in time and sets TQ_DEV_WAIT_TIMEOUT when it gives up.
#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"
#include "tmap.cuh"
#include "umma.cuh"

namespace tq {
namespace fa {

constexpr int kWarps = 8;                  // consumer warps, 16 query rows each
constexpr int kRows = kWarps * 16;         // query rows per CTA
constexpr int kTile = 64;                  // keys per stage
constexpr int kSub = 32;                   // keys per TMA box
constexpr int kNS = 3;                     // stages
constexpr int kThreads = (kWarps + 1) * 32;
static_assert(kRows == kFlashRows, "the row-wise kernel skips blocks of kFlashRows / G rows");
constexpr uint64_t kWaitNs = 1000000000ull;

template <int HD>
struct Smem {
  static constexpr int HALVES = HD / 64;                  // 64-dimension halves of a key row
  static constexpr int BOX = kSub * 128;                  // one box: 32 keys x 64 dims
  static constexpr int TILE = HALVES * 2 * BOX;           // K or V of 64 keys
  static constexpr int STAGE = 2 * TILE;
  static constexpr int BYTES = 1024 + kNS * STAGE + 128;
};

#define kNegInf (-__int_as_float(0x7f800000))

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// hi: x with its low 13 mantissa bits cleared (exact in fp16 for |x| in the
// scaled range), lo: fp16(x - hi)
__device__ __forceinline__ float hi_part(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// Shared address of the 16-byte chunk c (dimensions 8c .. 8c + 7) of key k
// in a K or V tile: box (half c / 8, sub-tile k / 32), row k % 32, chunk
// swizzled by the row's low three bits.
template <int HD>
__device__ __forceinline__ uint32_t chunk_addr(uint32_t tile, int k, int c) {
  return tile + (uint32_t)(((c >> 3) * 2 + (k >> 5)) * Smem<HD>::BOX + (k & 31) * 128 + (((c & 7) ^ (k & 7)) << 4));
}

template <int HD, int G>
__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ AttnArgs a) {
  using S = Smem<HD>;
  constexpr int BQ = kRows / G;   // query tokens per CTA
  constexpr int KS = HD / 16;     // k-steps of the score MMA
  constexpr int ND = HD / 8;      // n-tiles of the output
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw0 = smem_addr(smem_raw);
  const uint32_t base = (raw0 + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw0);
  uint64_t* full = reinterpret_cast<uint64_t*>(sbase + kNS * S::STAGE);
  uint64_t* empty = full + kNS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kNS);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nqb = (a.T + BQ - 1) / BQ;
  const int qb = nqb - 1 - (int)blockIdx.x;  // longest prefixes first
  const int h = blockIdx.y;
  const int t0 = qb * BQ;
  const int t_last = min(a.T, t0 + BQ) - 1;
  // rows of a mixed step (seq_idx set): this block only when it is one
  // sequence's consecutive positions (every warp reaches the same answer);
  // the row-wise decode kernel takes the other rows
  int seq = a.seq_fixed, pos_base = a.pos_base;
  if (a.seq_idx != nullptr) {
    if (a.kv_len == nullptr || !rows_uniform(a.seq_idx, a.kv_len, t0, t_last + 1 - t0, a.cache)) return;
    seq = a.seq_idx[t0];
    pos_base = a.kv_len[t0] - t0;
  }
  const int n_keys = min(pos_base + t_last + 1, a.cache.max_ctx);
  const int n_tiles = (n_keys + kTile - 1) / kTile;
  // sliding window: tiles before the first key any query row of the CTA sees
  // are skipped (the rows' own lower bounds are masked below)
  const int i0 = a.window > 0 ? min(max(0, pos_base + t0 + 1 - a.window), n_keys) / kTile : 0;

  // zero the stages once: a box that is not loaded (past the prefix) then
  // holds finite values, which the mask turns into p = 0
  for (int i = tid; i < kNS * S::STAGE / 16; i += kThreads)
    reinterpret_cast<uint4*>(sbase)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async();  // these stores, before the TMA engine writes the same bytes
  if (tid == 0) {
    for (int k = 0; k < kNS; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], kWarps);
    }
    *abort_flag = 0;
    fence_proxy_async();
  }
  __syncthreads();
  grid_dep_launch();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      umma::prefetch_tmap(&kmap);
      umma::prefetch_tmap(&vmap);
      grid_dep_wait();  // the append kernel wrote this prompt's K/V rows
      int issued = 0;
      for (int i = i0; i < n_tiles; ++i) {
        const int ii = i - i0, slot = ii % kNS;  // stage ring position
        if (ii >= kNS && !mbar_wait_timed(&empty[slot], (uint32_t)(((ii / kNS) - 1) & 1), kWaitNs)) {
          set_status(a.status, TQ_DEV_WAIT_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        // boxes of this tile: sub-tiles that hold a key of the prefix
        int page[2] = {0, 0};
        bool ok[2] = {false, false};
        for (int st = 0; st < 2; ++st) {
          const int j0 = i * kTile + st * kSub;
          if (j0 >= n_keys) continue;
          if (a.cache.page_size > 0) {
            const int p = a.cache.block_table[(int64_t)seq * a.cache.bt_stride + j0 / a.cache.page_size];
            if (p < 0 || p >= a.cache.n_pages) {
              set_status(a.status, TQ_DEV_KV_OVERFLOW);
              continue;
            }
            page[st] = p;
          }
          ok[st] = true;
        }
        const uint32_t bytes = (uint32_t)((ok[0] + ok[1]) * S::HALVES * 2 * S::BOX);
        uint8_t* kt = sbase + slot * S::STAGE;
        uint8_t* vt = kt + S::TILE;
        mbar_arrive_expect_tx(&full[slot], bytes);
        for (int st = 0; st < 2; ++st) {
          if (!ok[st]) continue;
          const int j0 = i * kTile + st * kSub;
          for (int dh = 0; dh < S::HALVES; ++dh) {
            const int off = (dh * 2 + st) * S::BOX;
            if (a.cache.page_size > 0) {
              const int jr = j0 % a.cache.page_size;
              umma::tma_load_4d(kt + off, &kmap, dh * 64, jr, h, page[st], &full[slot]);
              umma::tma_load_4d(vt + off, &vmap, dh * 64, jr, h, page[st], &full[slot]);
            } else {
              umma::tma_load_3d(kt + off, &kmap, dh * 64, j0, seq * a.nkv + h, &full[slot]);
              umma::tma_load_3d(vt + off, &vmap, dh * 64, j0, seq * a.nkv + h, &full[slot]);
            }
          }
        }
        ++issued;
      }
      // every issued load lands before the CTA's shared memory is released
      for (int i = (issued > kNS ? issued - kNS : 0); i < issued; ++i)
        mbar_wait_timed(&full[i % kNS], (uint32_t)((i / kNS) & 1), kWaitNs);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const int ra = warp * 16 + g, rb = ra + 8;  // this thread's two query rows
  const int tok_a = t0 + ra / G, tok_b = t0 + rb / G;
  const int ha = h * G + ra % G, hb = h * G + rb % G;
  // rows past the prompt compute on zeros and are not written
  const int pos_a = pos_base + min(tok_a, t_last), pos_b = pos_base + min(tok_b, t_last);
  const int pmax = pos_base + min(t0 + (warp * 16 + 15) / G, t_last);
  // key j is visible to a row at position p iff lo < j <= p (lo = p - window, or -1)
  const int lo_a = a.window > 0 ? pos_a - a.window : -1, lo_b = a.window > 0 ? pos_b - a.window : -1;

  grid_dep_wait();  // q was normalised and rotated by the append kernel
  // ---- Q: both rows as fp16 hi/lo A fragments after a power-of-two scale
  uint32_t qh[KS][4], ql[KS][4];
  float mult_a, mult_b;
  {
    float xa[KS][4], xb[KS][4];
    const float* qa = a.q + (int64_t)tok_a * a.q_stride + ha * HD;
    const float* qbp = a.q + (int64_t)tok_b * a.q_stride + hb * HD;
    float ma = 0.f, mb = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = 16 * ks + 2 * c, d1 = d0 + 8;
      float2 v0 = make_float2(0.f, 0.f), v1 = v0, w0 = v0, w1 = v0;
      if (tok_a < a.T) {
        v0 = *reinterpret_cast<const float2*>(qa + d0);
        v1 = *reinterpret_cast<const float2*>(qa + d1);
      }
      if (tok_b < a.T) {
        w0 = *reinterpret_cast<const float2*>(qbp + d0);
        w1 = *reinterpret_cast<const float2*>(qbp + d1);
      }
      xa[ks][0] = v0.x; xa[ks][1] = v0.y; xa[ks][2] = v1.x; xa[ks][3] = v1.y;
      xb[ks][0] = w0.x; xb[ks][1] = w0.y; xb[ks][2] = w1.x; xb[ks][3] = w1.y;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ma = fmaxf(ma, fabsf(xa[ks][e]));
        mb = fmaxf(mb, fabsf(xb[ks][e]));
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {  // the quad holds the row
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, o));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    }
    auto exp_of = [](float mx) {  // 2^e puts mx in [2^14, 2^15)
      int e = 0;
      if (mx > 0.f && mx <= 3.4e38f) e = 14 - (int)((__float_as_uint(mx) >> 23) & 0xffu) + 127;
      return max(-100, min(100, e));
    };
    const int ea = exp_of(ma), eb = exp_of(mb);
    const float fa = __uint_as_float((uint32_t)(ea + 127) << 23), fb = __uint_as_float((uint32_t)(eb + 127) << 23);
    mult_a = __uint_as_float((uint32_t)(127 - ea) << 23) * a.scale_log2;
    mult_b = __uint_as_float((uint32_t)(127 - eb) << 23) * a.scale_log2;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      float sa[4], sb[4], ha4[4], hb4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sa[e] = xa[ks][e] * fa;
        sb[e] = xb[ks][e] * fb;
        ha4[e] = hi_part(sa[e]);
        hb4[e] = hi_part(sb[e]);
      }
      qh[ks][0] = pack_h2(ha4[0], ha4[1]);
      qh[ks][1] = pack_h2(hb4[0], hb4[1]);
      qh[ks][2] = pack_h2(ha4[2], ha4[3]);
      qh[ks][3] = pack_h2(hb4[2], hb4[3]);
      ql[ks][0] = pack_h2(sa[0] - ha4[0], sa[1] - ha4[1]);
      ql[ks][1] = pack_h2(sb[0] - hb4[0], sb[1] - hb4[1]);
      ql[ks][2] = pack_h2(sa[2] - ha4[2], sa[3] - ha4[3]);
      ql[ks][3] = pack_h2(sb[2] - hb4[2], sb[3] - hb4[3]);
    }
  }

  float o[ND][4];
#pragma unroll
  for (int nd = 0; nd < ND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;

  for (int i = i0; i < n_tiles; ++i) {
    const int ii = i - i0, slot = ii % kNS;
    bool ok = *abort_flag == 0 && mbar_wait_timed(&full[slot], (uint32_t)((ii / kNS) & 1), kWaitNs);
    if (!__all_sync(0xffffffffu, ok) && lane == 0 && *abort_flag == 0) {
      set_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      *abort_flag = 1;
    }
    const int key0 = i * kTile;
    if (key0 <= pmax) {
      const uint32_t kt = base + slot * S::STAGE, vt = kt + S::TILE;
      // ---- S = Q K^T (8 n-tiles of 8 keys)
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          // matrices: (n-tile 2np, dims lo), (2np, hi), (2np+1, lo), (2np+1, hi)
          const int mtx = lane >> 3;
          const int key = 8 * (2 * np + (mtx >> 1)) + (lane & 7);
          uint32_t b[4];
          ldsm_x4(chunk_addr<HD>(kt, key, 2 * ks + (mtx & 1)), b);
          mma(s[2 * np], qh[ks], b[0], b[1]);
          mma(s[2 * np], ql[ks], b[0], b[1]);
          mma(s[2 * np + 1], qh[ks], b[2], b[3]);
          mma(s[2 * np + 1], ql[ks], b[2], b[3]);
        }
      }
      // ---- mask, online softmax (base 2)
      float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int j = key0 + 8 * nt + 2 * c;
        s[nt][0] = j <= pos_a && j > lo_a ? s[nt][0] * mult_a : kNegInf;
        s[nt][1] = j + 1 <= pos_a && j + 1 > lo_a ? s[nt][1] * mult_a : kNegInf;
        s[nt][2] = j <= pos_b && j > lo_b ? s[nt][2] * mult_b : kNegInf;
        s[nt][3] = j + 1 <= pos_b && j + 1 > lo_b ? s[nt][3] * mult_b : kNegInf;
        mx_a = fmaxf(mx_a, fmaxf(s[nt][0], s[nt][1]));
        mx_b = fmaxf(mx_b, fmaxf(s[nt][2], s[nt][3]));
      }
#pragma unroll
      for (int o2 = 1; o2 <= 2; o2 <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o2));
      }
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float cr_a = m_a == kNegInf ? 0.f : exp2f(m_a - mn_a);
      const float cr_b = m_b == kNegInf ? 0.f : exp2f(m_b - mn_b);
      m_a = mn_a;
      m_b = mn_b;
      uint32_t p[4][4];  // A fragments of P, k-steps of 16 keys
      float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float p0 = s[nt][0] == kNegInf ? 0.f : exp2f(s[nt][0] - mn_a);
        const float p1 = s[nt][1] == kNegInf ? 0.f : exp2f(s[nt][1] - mn_a);
        const float p2 = s[nt][2] == kNegInf ? 0.f : exp2f(s[nt][2] - mn_b);
        const float p3 = s[nt][3] == kNegInf ? 0.f : exp2f(s[nt][3] - mn_b);
        sum_a += p0 + p1;
        sum_b += p2 + p3;
        p[nt >> 1][(nt & 1) * 2] = pack_h2(p0, p1);
        p[nt >> 1][(nt & 1) * 2 + 1] = pack_h2(p2, p3);
      }
      l_a = l_a * cr_a + sum_a;
      l_b = l_b * cr_b + sum_b;
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        o[nd][0] *= cr_a;
        o[nd][1] *= cr_a;
        o[nd][2] *= cr_b;
        o[nd][3] *= cr_b;
      }
      // ---- O += P V (4 k-steps of 16 keys)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int dp = 0; dp < ND / 2; ++dp) {
          // matrices: (keys lo, dims 2dp), (keys hi, 2dp), (keys lo, 2dp+1), (keys hi, 2dp+1)
          const int mtx = lane >> 3;
          const int key = 16 * kk + 8 * (mtx & 1) + (lane & 7);
          uint32_t b[4];
          ldsm_x4_t(chunk_addr<HD>(vt, key, 2 * dp + (mtx >> 1)), b);
          mma(o[2 * dp], p[kk], b[0], b[1]);
          mma(o[2 * dp + 1], p[kk], b[2], b[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // the producer may refill the stage
  }

  // ---- finish: the quad's row sums, O / l
#pragma unroll
  for (int o2 = 1; o2 <= 2; o2 <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, o2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, o2);
  }
  const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
  float* oa = a.o + (int64_t)tok_a * a.nq * HD + ha * HD;
  float* ob = a.o + (int64_t)tok_b * a.nq * HD + hb * HD;
#pragma unroll
  for (int nd = 0; nd < ND; ++nd) {
    const int d = 8 * nd + 2 * c;
    if (tok_a <= t_last) *reinterpret_cast<float2*>(oa + d) = make_float2(o[nd][0] * ia, o[nd][1] * ia);
    if (tok_b <= t_last) *reinterpret_cast<float2*>(ob + d) = make_float2(o[nd][2] * ib, o[nd][3] * ib);
  }
}

}  // namespace fa

// Tensor maps of one layer's K or V cache for attn_prefill: boxes of 32 keys
// x 64 dimensions.  Contiguous cache: dims {hd, max_ctx, max_batch * n_kv};
// paged: {hd, page_size, n_kv, n_pages}.
cudaError_t encode_kv_map(CUtensorMap* map, const void* layer_base, int hd, const CacheView& c, int max_batch) {
  if (c.page_size > 0) {
    const cuuint64_t dims[4] = {(cuuint64_t)hd, (cuuint64_t)c.page_size, (cuuint64_t)c.n_kv, (cuuint64_t)c.n_pages};
    const cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)c.page_size * hd * 2,
                                   (cuuint64_t)c.n_kv * c.page_size * hd * 2};
    const cuuint32_t box[4] = {64u, (cuuint32_t)fa::kSub, 1u, 1u};
    return tmap_f16_sw128(map, layer_base, 4, dims, strides, box);
  }
  const cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)c.max_ctx, (cuuint64_t)max_batch * c.n_kv};
  const cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)c.max_ctx * hd * 2};
  const cuuint32_t box[3] = {64u, (cuuint32_t)fa::kSub, 1u};
  return tmap_f16_sw128(map, layer_base, 3, dims, strides, box);
}

namespace {
template <int HD, int G>
cudaError_t launch_fa(const CUtensorMap& km, const CUtensorMap& vm, const AttnArgs& a, cudaStream_t s) {
  using S = fa::Smem<HD>;
  static PerDevice setup;
  cudaError_t e = per_device(setup, nullptr, [](int, int&) {
    return cudaFuncSetAttribute(fa::attn_prefill_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                S::BYTES);
  });
  if (e != cudaSuccess) return e;
  constexpr int BQ = fa::kRows / G;
  dim3 grid((a.T + BQ - 1) / BQ, a.nkv, 1);
  return launch_k(fa::attn_prefill_kernel<HD, G>, grid, dim3(fa::kThreads), S::BYTES, s, km, vm, a);
}
template <int HD>
cudaError_t launch_fa_h(int G, const CUtensorMap& km, const CUtensorMap& vm, const AttnArgs& a, cudaStream_t s) {
  switch (G) {
    case 1: return launch_fa<HD, 1>(km, vm, a, s);
    case 2: return launch_fa<HD, 2>(km, vm, a, s);
    case 4: return launch_fa<HD, 4>(km, vm, a, s);
    case 8: return launch_fa<HD, 8>(km, vm, a, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_attn_prefill(int hd, int G, const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a,
                                cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.seq_fixed < 0 && a.seq_idx == nullptr) return cudaErrorInvalidValue;
  return hd == 128 ? launch_fa_h<128>(G, kmap, vmap, a, s) : launch_fa_h<64>(G, kmap, vmap, a, s);
}

}  // namespace tq
