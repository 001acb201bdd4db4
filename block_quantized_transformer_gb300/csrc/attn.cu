// Attention side of the decode step ("Всередині LLM: чисте виконання на
// Python для Qwen3-0.6B на MLX", step 4 and step 5 "Вся функція уваги";
// "Inferencia local y arquitecturas", qwen3.archdef: norm_heads before rope):
//
//  * rope_append: per-head RMSNorm of every Q and K head over head_dim with
//    its gain, half-split RoPE from a host-made f32 cos/sin table, Q written
//    back in place, K (normed, rotated) and V converted to the cache type
//    (f16: round to nearest even) and stored at the token's cache index.
//  * attn_decode: split-K flash-decode grouped-query attention.  One CTA per
//    (split of the context, KV head, token); its four warps take 32-key tiles
//    of the split in turn.  Each tile's K and V rows are contiguous in the
//    cache and are staged into shared memory by the TMA engine (1-D bulk
//    copies completing on an mbarrier, no multicast).  The whole query group
//    (G heads sharing the KV head) is evaluated against each staged tile:
//    lane l owns head_dim/32 consecutive dimensions, partial dot products are
//    combined with a reduce-scatter butterfly that leaves lane l holding the
//    score of (head l / (32/G), key l % (32/G)), and an online softmax in base
//    2 keeps (max, sum, output) per head.  Warps merge in shared memory; the
//    CTA writes its split's partial (o, m, l); the last CTA of a (token, head)
//    to finish (atomic counter, no waiting) merges all splits and resets the
//    counter.
#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace tq {
namespace {

#define kNegInf (-__int_as_float(0x7f800000))
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kCluster = 16;  // CTAs per (token, KV head) in decode

template <typename KT>
__device__ __forceinline__ KT to_kv(float v);
template <>
__device__ __forceinline__ float to_kv<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half to_kv<__half>(float v) { return __float2half_rn(v); }

// Pointer to element 0 of cache row `slot` of (seq, kv head h), or null when
// the sequence, the slot or the page is out of range.
template <typename KT, int HD>
__device__ __forceinline__ KT* cache_row(void* base, int seq, int h, int slot, const CacheView& c) {
  if (seq < 0 || seq >= c.max_seq) return nullptr;
  if (slot < 0 || slot >= c.max_ctx) return nullptr;
  if (c.page_size == 0) {
    return reinterpret_cast<KT*>(base) + (((int64_t)seq * c.n_kv + h) * c.max_ctx + slot) * HD;
  }
  const int page = c.block_table[(int64_t)seq * c.bt_stride + slot / c.page_size];
  if (page < 0 || page >= c.n_pages) return nullptr;
  return reinterpret_cast<KT*>(base) +
         (((int64_t)page * c.n_kv + h) * c.page_size + slot % c.page_size) * HD;
}

template <typename KT, int HD>
__global__ void __launch_bounds__(128) rope_append_kernel(RopeArgs a) {
  constexpr int DPL = HD / 32;
  grid_dep_launch();
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hi = blockIdx.x * 4 + warp;
  const int t = blockIdx.y;
  if (hi >= a.nq + a.nkv) return;
  const int pos = a.pos != nullptr ? a.pos[t] : a.pos_base + t;
  const int slot = a.kv_len != nullptr ? a.kv_len[t] : a.pos_base + t;
  const int seq = a.seq_idx != nullptr ? a.seq_idx[t] : a.seq_fixed >= 0 ? a.seq_fixed : t;
  const int row_stride = (a.nq + 2 * a.nkv) * HD;
  float* row = a.qkv + (int64_t)t * row_stride;
  const bool is_q = hi < a.nq;
  float* src = row + (is_q ? hi * HD : a.nq * HD + (hi - a.nq) * HD);

  float x[DPL];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    x[j] = src[lane + 32 * j];
    ss = fmaf(x[j], x[j], ss);
  }
  const float* g = is_q ? a.gq : a.gk;
  if (g != nullptr) {  // per-head RMSNorm (absent from some layer recipes)
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)HD + a.eps);
#pragma unroll
    for (int j = 0; j < DPL; ++j) x[j] = x[j] * inv * g[lane + 32 * j];
  }

  if (pos >= 0 && pos < a.cache.max_ctx) {
    constexpr int HALF = HD / 2;
#pragma unroll
    for (int j = 0; j < DPL / 2; ++j) {
      const int i = lane + 32 * j;
      const float c = a.cos_t[(int64_t)pos * HALF + i];
      const float s = a.sin_t[(int64_t)pos * HALF + i];
      const float x1 = x[j], x2 = x[j + DPL / 2];
      x[j] = x1 * c - x2 * s;
      x[j + DPL / 2] = x1 * s + x2 * c;
    }
  } else if (lane == 0) {
    set_status(a.status, TQ_DEV_KV_OVERFLOW);
  }

  if (is_q) {
#pragma unroll
    for (int j = 0; j < DPL; ++j) src[lane + 32 * j] = x[j];
    return;
  }
  const int h = hi - a.nq;
  KT* kd = cache_row<KT, HD>(a.kc, seq, h, slot, a.cache);
  KT* vd = cache_row<KT, HD>(a.vc, seq, h, slot, a.cache);
  if (kd == nullptr || vd == nullptr) {
    if (lane == 0) set_status(a.status, TQ_DEV_KV_OVERFLOW);
    return;
  }
  const float* vsrc = row + (a.nq + a.nkv) * HD + h * HD;
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    kd[lane + 32 * j] = to_kv<KT>(x[j]);
    vd[lane + 32 * j] = to_kv<KT>(vsrc[lane + 32 * j]);
  }
}

// ------------------------------------------------------------ attention --

template <typename KT, int DPL>
__device__ __forceinline__ void load_row(const KT* p, float (&v)[DPL]);
template <>
__device__ __forceinline__ void load_row<__half, 4>(const __half* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
template <>
__device__ __forceinline__ void load_row<__half, 2>(const __half* p, float (&v)[2]) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
  v[0] = a.x; v[1] = a.y;
}
template <>
__device__ __forceinline__ void load_row<float, 4>(const float* p, float (&v)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
template <>
__device__ __forceinline__ void load_row<float, 2>(const float* p, float (&v)[2]) {
  const float2 a = *reinterpret_cast<const float2*>(p);
  v[0] = a.x; v[1] = a.y;
}

// RMSNorm over the head (gain g; skipped when !norm) and half-split RoPE at `pos` of one head held
// as DPL consecutive dimensions per lane (lane l: dims l*DPL ..): the partner
// of dimension i < hd/2 is i + hd/2, which lives in lane l ^ 16.
template <int HD, int DPL>
__device__ __forceinline__ void norm_rope_head(float (&x)[DPL], const float (&g)[DPL], float eps,
                                               const float (&c)[DPL], const float (&sn)[DPL],
                                               int lane, bool rope_ok, bool norm) {
  if (norm) {
    float ss = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) ss = fmaf(x[d], x[d], ss);
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
    for (int d = 0; d < DPL; ++d) x[d] = x[d] * inv * g[d];
  }
  if (!rope_ok) return;
  const bool first = lane < 16;
#pragma unroll
  for (int d = 0; d < DPL; ++d) {
    const float other = __shfl_xor_sync(0xffffffffu, x[d], 16);
    x[d] = first ? x[d] * c[d] - other * sn[d] : other * sn[d] + x[d] * c[d];
  }
}

// reduce-scatter of 32 values over a full warp: lane l ends with sum of v[l]
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < n / 2) {
        const float send = upper ? v[i] : v[i + n / 2];
        const float keep = upper ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  return v[0];
}

template <typename KT, int HD, int G, int NS>
struct AttnSmem {
  // res_*: this CTA's merged (m, l, o) read by the cluster's rank 0
  static constexpr int TILE = 32;
  static constexpr int TILE_BYTES = TILE * HD * (int)sizeof(KT);
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = 4 * NS * STAGE_BYTES;
  static constexpr int OFF_P = OFF_BAR + 4 * NS * 8;
  static constexpr int OFF_ALPHA = OFF_P + 4 * G * 32 * 4;
  static constexpr int OFF_M = OFF_ALPHA + 4 * G * 4;
  static constexpr int OFF_L = OFF_M + 4 * G * 4;
  static constexpr int OFF_O = OFF_L + 4 * G * 4;
  static constexpr int OFF_FLAG = OFF_O + 4 * G * HD * 4;
  static constexpr int OFF_RES = OFF_FLAG + 16;
  static constexpr int BYTES = OFF_RES + (2 * G + G * HD) * 4;
};

// FUSED (decode): q arrives straight from the Q/K/V projection; each CTA
// applies QK-RMSNorm and RoPE to its query group itself, and the warp whose
// tile holds the new position computes the new K (normed, rotated) and V,
// stores them in the cache and only then stages that tile.  Older cache
// positions are read-only in this step, so their tiles are staged before
// waiting for the preceding kernel.
// CL > 0: the CL CTAs of a cluster split the context of one (token, KV head)
// evenly at run time and merge through distributed shared memory: no
// partials in global memory, no counters, no fences.  CL == 0: fixed-size
// splits merged by the last CTA to finish, through global memory.
template <typename KT, int HD, int G, int NS, bool FUSED, int CL>
__global__ void __launch_bounds__(128) attn_decode_kernel(AttnArgs a) {
  using S = AttnSmem<KT, HD, G, NS>;
  constexpr int DPL = HD / 32;
  constexpr int CK = 32 / G;     // keys per score chunk
  constexpr int NCH = 32 / CK;   // chunks per tile (= G)
  constexpr int TILE = S::TILE;
  extern __shared__ __align__(128) uint8_t smem[];

  grid_dep_launch();
  const int split = blockIdx.x, h = blockIdx.y, t = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  if (!FUSED) grid_dep_wait();
  // kv_len is an input of the step, never written by a kernel of the step
  const int new_slot = a.kv_len != nullptr ? a.kv_len[t] : a.pos_base + t;
  int ctx = new_slot + 1;
  if (ctx > a.cache.max_ctx) ctx = a.cache.max_ctx;
  // sliding window: keys lo .. ctx - 1, split from lo rounded down to a tile
  const int lo = a.window > 0 ? max(0, new_slot + 1 - a.window) : 0;
  const int lo_t = (min(lo, ctx - 1) / TILE) * TILE;
  // cluster: keys per CTA rounded up to whole tiles
  const int span = CL > 0 ? ((ctx - lo_t + CL * TILE - 1) / (CL * TILE)) * TILE : a.split_keys;
  const int n_active = (ctx - lo_t + span - 1) / span;
  if (CL == 0 && split >= n_active) return;
  const int seq = a.seq_idx != nullptr ? a.seq_idx[t] : a.seq_fixed >= 0 ? a.seq_fixed : t;
  const int k0 = lo_t + split * span;
  const int k1 = min(ctx, k0 + span);
  const int n_tiles = k1 > k0 ? (k1 - k0 + TILE - 1) / TILE : 0;
  const int my_n = warp < n_tiles ? (n_tiles - warp + 3) / 4 : 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR) + warp * NS;
  float* p_s = reinterpret_cast<float*>(smem + S::OFF_P) + warp * G * 32;
  float* alpha_s = reinterpret_cast<float*>(smem + S::OFF_ALPHA) + warp * G;
  float* m_s = reinterpret_cast<float*>(smem + S::OFF_M);
  float* l_s = reinterpret_cast<float*>(smem + S::OFF_L);
  float* o_s = reinterpret_cast<float*>(smem + S::OFF_O);
  int* flag_s = reinterpret_cast<int*>(smem + S::OFF_FLAG);

  const int gl = lane / CK;  // the head whose scores this lane holds
  float m_run = kNegInf, l_run = 0.f;
  float o[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[g][d] = 0.f;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_proxy_async();
  }
  __syncwarp();

  auto tile_key0 = [&](int k) { return k0 + (warp + 4 * k) * TILE; };
  auto issue = [&](int k) {
    const int key0 = tile_key0(k);
    const int nv = min(TILE, k1 - key0);
    const uint32_t bytes = (uint32_t)(nv * HD * sizeof(KT));
    const KT* ks = cache_row<KT, HD>(const_cast<void*>(a.kc), seq, h, key0, a.cache);
    const KT* vs = cache_row<KT, HD>(const_cast<void*>(a.vc), seq, h, key0, a.cache);
    uint8_t* st = smem + ((warp * NS + k % NS) * S::STAGE_BYTES);
    if (ks == nullptr || vs == nullptr) {
      // unreachable for in-range slots; keep the barrier phase moving
      set_status(a.status, TQ_DEV_KV_OVERFLOW);
      mbar_arrive_expect_tx(&bars[k % NS], 0);
      return;
    }
    mbar_arrive_expect_tx(&bars[k % NS], 2 * bytes);
    bulk_g2s(st, ks, bytes, &bars[k % NS]);
    bulk_g2s(st + S::TILE_BYTES, vs, bytes, &bars[k % NS]);
  };
  // the warp whose last tile holds the new position (FUSED only)
  const bool owns_new = FUSED && my_n > 0 && new_slot >= k0 && new_slot < k1 &&
                        ((new_slot - k0) / TILE) % 4 == warp;
  // Read-only inputs first (cache tiles of earlier positions, gains, the RoPE
  // row of this position), all before waiting for the preceding kernel.
  if (FUSED && lane == 0)
    for (int k = 0; k < NS && k < my_n; ++k)
      if (!(owns_new && k == my_n - 1)) issue(k);
  const int pos = FUSED ? a.pos[t] : 0;
  const bool rope_ok = pos >= 0 && pos < a.cache.max_ctx;
  float gq[DPL], gk[DPL], cs[DPL], sn[DPL];
  if (FUSED) {
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      const int i = (lane * DPL + d) % (HD / 2);
      gq[d] = a.gq != nullptr ? a.gq[lane * DPL + d] : 1.f;
      gk[d] = a.gk != nullptr ? a.gk[lane * DPL + d] : 1.f;
      cs[d] = rope_ok ? a.cos_t[(int64_t)pos * (HD / 2) + i] : 1.f;
      sn[d] = rope_ok ? a.sin_t[(int64_t)pos * (HD / 2) + i] : 0.f;
    }
    if (!rope_ok && tid == 0) set_status(a.status, TQ_DEV_KV_OVERFLOW);
    grid_dep_wait();
  }
  if (!FUSED && lane == 0)
    for (int k = 0; k < NS && k < my_n; ++k) issue(k);

  // query group (and the new K/V), loaded together, normed, rotated and
  // pre-scaled into the base-2 softmax domain
  const float* qrow = a.q + (int64_t)t * a.q_stride;
  float qr[G][DPL], kx[DPL], vx[DPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float* qp = qrow + (h * G + g) * HD + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; ++d) qr[g][d] = qp[d];
  }
  if (owns_new) {
    const float* kp = qrow + (a.nq + h) * HD + lane * DPL;
    const float* vp = qrow + (a.nq + a.nkv + h) * HD + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      kx[d] = kp[d];
      vx[d] = vp[d];
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (FUSED) norm_rope_head<HD, DPL>(qr[g], gq, a.eps, cs, sn, lane, rope_ok, a.gq != nullptr);
#pragma unroll
    for (int d = 0; d < DPL; ++d) qr[g][d] *= a.scale_log2;
  }
  if (owns_new) {
    norm_rope_head<HD, DPL>(kx, gk, a.eps, cs, sn, lane, rope_ok, a.gk != nullptr);
    KT* kd = cache_row<KT, HD>(const_cast<void*>(a.kc), seq, h, new_slot, a.cache);
    KT* vd = cache_row<KT, HD>(const_cast<void*>(a.vc), seq, h, new_slot, a.cache);
    if (kd != nullptr && vd != nullptr) {
#pragma unroll
      for (int d = 0; d < DPL; ++d) {
        kd[lane * DPL + d] = to_kv<KT>(kx[d]);
        vd[lane * DPL + d] = to_kv<KT>(vx[d]);
      }
    } else if (lane == 0) {
      set_status(a.status, TQ_DEV_KV_OVERFLOW);
    }
    fence_proxy_async_global();  // the new row is read back by the TMA engine
    __syncwarp();
    if (lane == 0 && my_n - 1 < NS) issue(my_n - 1);
  }

  bool failed = false;
  int consumed = 0;
  for (int k = 0; k < my_n; ++k) {
    const int stage = k % NS;
    // every lane waits: the warp sleeps in the barrier instead of one lane spinning
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[stage], (uint32_t)((k / NS) & 1), kWaitLimit));
    if (!ok) {
      if (lane == 0) set_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      failed = true;
      break;
    }
    consumed = k + 1;
    const KT* Ks = reinterpret_cast<const KT*>(smem + (warp * NS + stage) * S::STAGE_BYTES);
    const KT* Vs = reinterpret_cast<const KT*>(smem + (warp * NS + stage) * S::STAGE_BYTES + S::TILE_BYTES);
    const int nv = min(TILE, k1 - tile_key0(k));
    const int nlo = lo - tile_key0(k);  // keys of the tile before the window

    // scores of the whole query group against the tile's keys
    float sc[NCH];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      float v[32];
#pragma unroll
      for (int j = 0; j < CK; ++j) {
        float kv[DPL];
        load_row<KT, DPL>(Ks + (c * CK + j) * HD + lane * DPL, kv);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float acc = 0.f;
#pragma unroll
          for (int d = 0; d < DPL; ++d) acc = fmaf(qr[g][d], kv[d], acc);
          v[g * CK + j] = acc;
        }
      }
      const float s = reduce_scatter32(v, lane);
      sc[c] = (c * CK + lane % CK) < nv && (c * CK + lane % CK) >= nlo ? s : kNegInf;
    }
    // online softmax for head gl
    float mt = sc[0];
#pragma unroll
    for (int c = 1; c < NCH; ++c) mt = fmaxf(mt, sc[c]);
#pragma unroll
    for (int off = CK / 2; off >= 1; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    const float m_new = fmaxf(m_run, mt);
    const float alpha = exp2f(m_run - m_new);
    float psum = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const float p = exp2f(sc[c] - m_new);
      psum += p;
      p_s[gl * 32 + c * CK + lane % CK] = p;
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    if (lane % CK == 0) alpha_s[gl] = alpha;
    __syncwarp();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float al = alpha_s[g];
#pragma unroll
      for (int d = 0; d < DPL; ++d) o[g][d] *= al;
    }
    for (int j = 0; j < nv; ++j) {
      float vv[DPL];
      load_row<KT, DPL>(Vs + j * HD + lane * DPL, vv);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = p_s[g * 32 + j];
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[g][d] = fmaf(p, vv[d], o[g][d]);
      }
    }
    __syncwarp();
    if (lane == 0 && k + NS < my_n) {
      fence_proxy_async();
      issue(k + NS);
    }
  }
  if (failed && lane == 0) {
    // let copies already in flight land before the shared memory is released
    for (int k = consumed; k < my_n && k < consumed + NS; ++k)
      mbar_wait_bounded(&bars[k % NS], (uint32_t)((k / NS) & 1), kWaitLimit);
  }

  // ---- merge the four warps
#pragma unroll
  for (int off = CK / 2; off >= 1; off >>= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
  if (lane % CK == 0) {
    m_s[warp * G + gl] = m_run;
    l_s[warp * G + gl] = l_run;
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < DPL; ++d) o_s[(warp * G + g) * HD + lane * DPL + d] = o[g][d];
  __syncthreads();

  if (CL > 0) {
    // this CTA's (m, l, o) into shared memory, then rank 0 merges the cluster
    float* res_m = reinterpret_cast<float*>(smem + S::OFF_RES);
    float* res_l = res_m + G;
    float* res_o = res_l + G;
    for (int i = tid; i < G * HD; i += 128) {
      const int g = i / HD, d = i % HD;
      float M = kNegInf;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, m_s[w * G + g]);
      float acc = 0.f, L = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float f = M == kNegInf ? 0.f : exp2f(m_s[w * G + g] - M);
        acc += f * o_s[(w * G + g) * HD + d];
        L += f * l_s[w * G + g];
      }
      res_o[i] = acc;
      if (d == 0) {
        res_m[g] = M;
        res_l[g] = L;
      }
    }
    cluster_sync_all();
    // every rank merges its 1/CL share of the G*HD outputs of the cluster
    constexpr int SHARE = (G * HD + CL - 1) / (CL > 0 ? CL : 1);
    for (int i = split * SHARE + tid; i < (split + 1) * SHARE && i < G * HD; i += 128) {
      const int g = i / HD;
      float mr[CL > 0 ? CL : 1];
      float M = kNegInf;
#pragma unroll
      for (int r = 0; r < CL; ++r) {
        mr[r] = ld_cluster_f32(map_cluster(res_m + g, r));
        M = fmaxf(M, mr[r]);
      }
      float acc = 0.f, L = 0.f;
#pragma unroll
      for (int r = 0; r < CL; ++r) {
        const float f = mr[r] == kNegInf ? 0.f : exp2f(mr[r] - M);
        acc += f * ld_cluster_f32(map_cluster(res_o + i, r));
        L += f * ld_cluster_f32(map_cluster(res_l + g, r));
      }
      a.o[(int64_t)t * a.nq * HD + (h * G) * HD + i] = acc / L;
    }
    cluster_sync_all();  // no CTA leaves while another rank still reads its shared memory
    return;
  }

  const int64_t th = (int64_t)t * a.nkv + h;
  float* part = a.part + (th * a.max_splits + split) * (G * (HD + 2));
  for (int i = tid; i < G * HD; i += 128) {
    const int g = i / HD, d = i % HD;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, m_s[w * G + g]);
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = exp2f(m_s[w * G + g] - M);
      acc += f * o_s[(w * G + g) * HD + d];
      L += f * l_s[w * G + g];
    }
    if (n_active == 1) {
      a.o[(int64_t)t * a.nq * HD + (h * G + g) * HD + d] = acc / L;
    } else {
      part[g * (HD + 2) + d] = acc;
      if (d == 0) {
        part[g * (HD + 2) + HD] = M;
        part[g * (HD + 2) + HD + 1] = L;
      }
    }
  }
  if (n_active == 1) return;

  // ---- the last split to finish merges all splits
  __threadfence();
  __syncthreads();
  if (tid == 0) flag_s[0] = (atomicAdd(a.counters + th, 1u) == (unsigned)(n_active - 1)) ? 1 : 0;
  __syncthreads();
  if (flag_s[0] == 0) return;
  __threadfence();
  const float* base = a.part + th * a.max_splits * (G * (HD + 2));
  for (int i = tid; i < G * HD; i += 128) {
    const int g = i / HD, d = i % HD;
    float M = kNegInf;
    for (int s = 0; s < n_active; ++s) M = fmaxf(M, __ldcg(base + (s * G + g) * (HD + 2) + HD));
    float acc = 0.f, L = 0.f;
    for (int s = 0; s < n_active; ++s) {
      const float* ps = base + (s * G + g) * (HD + 2);
      const float f = exp2f(__ldcg(ps + HD) - M);
      acc += f * __ldcg(ps + d);
      L += f * __ldcg(ps + HD + 1);
    }
    a.o[(int64_t)t * a.nq * HD + (h * G + g) * HD + d] = acc / L;
  }
  if (tid == 0) a.counters[th] = 0u;
}

// ------------------------------------------------- tensor-core decode path --
//
// Fused decode over an f16 cache with the products on the tensor cores.  Same
// split of work, prologue (QK-norm, RoPE, append) and cluster merge as
// attn_decode_kernel<__half, .., FUSED, kCluster>; per 32-key tile:
//  * the warp's lane 0 stages K and V through the layer's tensor maps (TMA:
//    boxes of 32 keys x 64 dimensions, 128-byte swizzle, one mbarrier per
//    buffer), so a key's 16-byte chunks are XOR-swizzled by its low three
//    bits and ldmatrix reads of eight keys hit eight different banks; V rows
//    past the context are zeroed once the tile has landed (p = 0 must meet
//    finite values);
//  * scores S^T = K Q^T with mma.m16n8k16: A = K rows (exact f16), B = the
//    query group, every head as an unevaluated sum hi + lo of two fp16 values
//    after a per-head power-of-two scale (columns 2h, 2h+1), f32 sums;
//  * online base-2 softmax per head on the score fragments (a thread holds
//    four keys of one head; three shuffles finish a tile);
//  * O^T += V^T P^T: A = V read with ldmatrix.trans, B = the probabilities,
//    again as hi + lo fp16 pairs of p * 2^14, f32 accumulators.
// Products are exact and sums f32, so the result matches the scalar path to
// f32 rounding.

template <int HD, int G, int CL>
struct TcSmem {
  static constexpr int TILE = 32;
  static constexpr int BOX = TILE * 128;                 // 32 keys x 64 dimensions
  static constexpr int TILE_BYTES = TILE * HD * 2;       // one K or V tile: HD / 64 boxes
  static constexpr int WARP_BYTES = 2 * TILE_BYTES;
  static constexpr int OFF_P = 4 * WARP_BYTES;           // [warp][G][32] probabilities
  static constexpr int OFF_Q = OFF_P + 4 * G * 32 * 4;   // [G][HD] scaled q
  static constexpr int OFF_QS = OFF_Q + G * HD * 4;      // [G] 1 / (q scale)
  static constexpr int OFF_M = OFF_QS + ((G * 4 + 15) / 16) * 16;
  static constexpr int OFF_L = OFF_M + 4 * G * 4;
  static constexpr int OFF_O = OFF_L + 4 * G * 4;
  static constexpr int OFF_RES = OFF_O + 4 * G * HD * 4;
  static constexpr int SHARE = G * HD / CL;              // outputs each cluster rank finishes
  static constexpr int OFF_IN = OFF_RES + (2 * G + G * HD) * 4;  // [rank][SHARE + 2G] pushed to this rank
  static constexpr int OFF_BAR = (OFF_IN + CL * (SHARE + 2 * G) * 4 + 15) / 16 * 16;  // [warp][K, V] mbarriers
  static constexpr int BYTES = OFF_BAR + 8 * 8 + 1024;   // + slack to align the tiles to 1024 bytes (swizzle atom)
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// hi = x with its low 13 mantissa bits cleared (exact in fp16 for |x| >= 2^-14),
// lo = fp16(x - hi); packs (hi or lo of a, of b) into an fp16 pair.
__device__ __forceinline__ uint32_t split_pair(float a, float b, bool lo_part) {
  const float ha = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
  const float hb = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
  const __half2 v = lo_part ? __floats2half2_rn(a - ha, b - hb) : __floats2half2_rn(ha, hb);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// FUSED (decode): q, k, v come unnormalised from the projection; QK-norm,
// RoPE and the append of the new row happen here, and the rows of earlier
// positions are staged before waiting for the projection.  Not FUSED
// (prefill): the append kernel already normalised and rotated q and stored
// every row's K/V, so nothing is staged before the wait; rows are taken
// longest prefix first.
// Shared-memory address of 16-byte chunk c (dimensions 8c .. 8c + 7) of key
// row `key` in a tile staged as 128-byte-swizzled boxes of 64 dimensions.
__device__ __forceinline__ uint32_t tile_chunk(uint32_t tile, int key, int c) {
  return tile + (uint32_t)((c >> 3) * (32 * 128) + key * 128 + (((c & 7) ^ (key & 7)) << 4));
}

template <int HD, int G, int CL, bool FUSED>
__global__ void __launch_bounds__(128) attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                      const __grid_constant__ CUtensorMap vmap, AttnArgs a) {
  using S = TcSmem<HD, G, CL>;
  constexpr int DPL = HD / 32;
  constexpr int TILE = S::TILE;
  constexpr int NT = G > 4 ? 2 : 1;        // n-tiles of 4 heads (8 columns: hi, lo)
  constexpr int KS = HD / 16;              // k-steps of the score MMA
  constexpr uint64_t kTileWaitNs = 1000000000ull;  // 1 s: far beyond any legitimate wait
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

  grid_dep_launch();
  const int split = blockIdx.x, h = blockIdx.y, t = FUSED ? blockIdx.z : gridDim.z - 1 - blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int g = lane >> 2, c = lane & 3;
  // mixed rows: a block that attn_prefill takes (one sequence's consecutive
  // positions) is not computed here (every warp, and every CTA of a cluster,
  // reaches the same answer)
  if (!FUSED && a.flash_rows && a.seq_idx != nullptr && a.kv_len != nullptr) {
    constexpr int BQ = kFlashRows / G;
    const int tb = (t / BQ) * BQ;
    if (rows_uniform(a.seq_idx, a.kv_len, tb, min(a.T, tb + BQ) - tb, a.cache)) return;
  }
  // step inputs, never written by a kernel of the step: load both at once
  const int new_slot = a.kv_len != nullptr ? a.kv_len[t] : a.pos_base + t;
  const int pos = FUSED ? a.pos[t] : 0;
  int ctx = new_slot + 1;
  if (ctx > a.cache.max_ctx) ctx = a.cache.max_ctx;
  // sliding window: keys lo .. ctx - 1, split from lo rounded down to a tile
  const int lo = a.window > 0 ? max(0, new_slot + 1 - a.window) : 0;
  const int lo_t = (min(lo, ctx - 1) / TILE) * TILE;
  const int span = ((ctx - lo_t + CL * TILE - 1) / (CL * TILE)) * TILE;
  // a sequence index outside the cache: reads stay in bounds (sequence 0),
  // the new row is not written, the status says so
  const int seq_in = a.seq_idx != nullptr ? a.seq_idx[t] : a.seq_fixed >= 0 ? a.seq_fixed : t;
  const bool seq_ok = seq_in >= 0 && seq_in < a.cache.max_seq;
  const int seq = seq_ok ? seq_in : 0;
  if (!seq_ok && tid == 0) set_status(a.status, TQ_DEV_KV_OVERFLOW);
  const int k0 = lo_t + split * span;
  const int k1 = min(ctx, k0 + span);
  const int n_tiles = k1 > k0 ? (k1 - k0 + TILE - 1) / TILE : 0;
  const int my_n = warp < n_tiles ? (n_tiles - warp + 3) / 4 : 0;

  uint8_t* kt = smem + warp * S::WARP_BYTES;
  uint8_t* vt = kt + S::TILE_BYTES;
  const uint32_t kt_s = smem_addr(kt), vt_s = smem_addr(vt);
  float* p_s = reinterpret_cast<float*>(smem + S::OFF_P) + warp * G * 32;
  float* q_s = reinterpret_cast<float*>(smem + S::OFF_Q);
  float* qs_s = reinterpret_cast<float*>(smem + S::OFF_QS);
  float* m_s = reinterpret_cast<float*>(smem + S::OFF_M);
  float* l_s = reinterpret_cast<float*>(smem + S::OFF_L);
  float* o_s = reinterpret_cast<float*>(smem + S::OFF_O);

  auto tile_key0 = [&](int k) { return k0 + (warp + 4 * k) * TILE; };
  uint64_t* kbar = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR) + 2 * warp;
  uint64_t* vbar = kbar + 1;
  if (lane == 0) {
    if (warp == 0) {
      umma::prefetch_tmap(&kmap);
      umma::prefetch_tmap(&vmap);
    }
    mbar_init(kbar, 1);
    mbar_init(vbar, 1);
    fence_proxy_async();
  }
  __syncwarp();
  // Stage the K (V) rows of tile k: lane 0 issues the tile's boxes through
  // the tensor map (a tile's 32 keys are consecutive rows of one page: pages
  // hold a multiple of 32 keys, tiles start at multiples of 32); a page
  // outside the pool stages nothing (its rows are zeroed after the wait).
  // Keys past max_ctx read as zeros; keys past the context are masked.
  bool stage_ok = true;  // false once a wait gave up: no copy is issued after that
  int pend_k = -1, pend_v = -1;  // parity of a K (V) wait that gave up: that copy may still land
  auto page_of = [&](int key0) {
    return a.cache.page_size > 0 ? a.cache.block_table[(int64_t)seq * a.cache.bt_stride + key0 / a.cache.page_size]
                                 : 0;
  };
  auto stage_one = [&](int k, bool is_v) {
    if (lane == 0 && stage_ok) {
      const int key0 = tile_key0(k);
      uint64_t* bar = is_v ? vbar : kbar;
      uint8_t* dst = is_v ? vt : kt;
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      const int page = page_of(key0);
      fence_proxy_async();  // this warp's reads (and zeroing) of the buffer come before the copy's writes
      if (page >= 0 && page < (a.cache.page_size > 0 ? a.cache.n_pages : 1)) {
        mbar_arrive_expect_tx(bar, (uint32_t)S::TILE_BYTES);
#pragma unroll
        for (int dh = 0; dh < HD / 64; ++dh) {
          if (a.cache.page_size > 0)
            umma::tma_load_4d(dst + dh * S::BOX, map, dh * 64, key0 % a.cache.page_size, h, page, bar);
          else
            umma::tma_load_3d(dst + dh * S::BOX, map, dh * 64, key0, seq * a.nkv + h, bar);
        }
      } else {
        mbar_arrive(bar);
      }
    }
  };
  auto stage = [&](int k) {
    stage_one(k, false);
    stage_one(k, true);
  };
  // wait for tile k of K (V); on a time-out the status is set and no further
  // copy is issued (the values are then garbage, the status says so)
  auto wait_tile = [&](int k, bool is_v) {
    if (!mbar_wait_timed(is_v ? vbar : kbar, (uint32_t)(k & 1), kTileWaitNs)) {
      if (lane == 0) set_status(a.status, TQ_DEV_WAIT_TIMEOUT);
      int& pend = is_v ? pend_v : pend_k;
      if (pend < 0) pend = k & 1;  // the buffer's one copy in flight
      stage_ok = false;
    }
    __syncwarp();
  };
  // rows [nvalid, 32) of a landed tile are zeroed (all of it for a page
  // outside the pool, so its keys score 0 against finite values)
  auto zero_rows = [&](uint8_t* buf, int k) {
    const int key0 = tile_key0(k);
    const int page = page_of(key0);
    const bool in_pool = page >= 0 && page < (a.cache.page_size > 0 ? a.cache.n_pages : 1);
    const int nvalid = in_pool ? min(TILE, k1 - key0) : 0;
    if (nvalid >= TILE) return;
    for (int i = lane; i < (TILE - nvalid) * (HD / 8); i += 32) {
      const int key = nvalid + i / (HD / 8), c = i % (HD / 8);
      *reinterpret_cast<uint4*>(buf + tile_chunk(0u, key, c)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();  // these writes, before a later tensor copy into the buffer
    __syncwarp();
  };
  const bool owns_new =
      FUSED && my_n > 0 && new_slot >= k0 && new_slot < k1 && ((new_slot - k0) / TILE) % 4 == warp;
  // decode: the first tile of earlier positions is read-only: staged before waiting
  if (FUSED && my_n > 0 && !(owns_new && my_n == 1)) stage(0);
  const bool rope_ok = pos >= 0 && pos < a.cache.max_ctx;
  float gq[DPL], gk[DPL], cs[DPL], sn[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) {
    const int i = (lane * DPL + d) % (HD / 2);
    gq[d] = FUSED && a.gq != nullptr ? a.gq[lane * DPL + d] : 1.f;
    gk[d] = FUSED && a.gk != nullptr ? a.gk[lane * DPL + d] : 1.f;
    cs[d] = FUSED && rope_ok ? a.cos_t[(int64_t)pos * (HD / 2) + i] : 1.f;
    sn[d] = FUSED && rope_ok ? a.sin_t[(int64_t)pos * (HD / 2) + i] : 0.f;
  }
  if (FUSED && !rope_ok && tid == 0) set_status(a.status, TQ_DEV_KV_OVERFLOW);
  grid_dep_wait();
  if (!FUSED && my_n > 0) stage(0);  // prefill: the rows were written by the preceding kernel

  // query group: warp w normalises, rotates and scales heads w, w+4 into q_s
  const float* qrow = a.q + (int64_t)t * a.q_stride;
  for (int gg = warp; gg < G; gg += 4) {
    float qr[DPL];
    const float* qp = qrow + (h * G + gg) * HD + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; ++d) qr[d] = qp[d];
    if (FUSED) norm_rope_head<HD, DPL>(qr, gq, a.eps, cs, sn, lane, rope_ok, a.gq != nullptr);
    float mx = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      qr[d] *= a.scale_log2;
      mx = fmaxf(mx, fabsf(qr[d]));
    }
    mx = warp_max(mx);
    int e2 = 0;  // scale the head so its largest |q| lies in [2^14, 2^15)
    if (mx > 0.f && mx <= 3.4e38f) e2 = 14 - (int)((__float_as_uint(mx) >> 23) & 0xffu) + 127;
    e2 = max(-100, min(100, e2));
    const float sc = __uint_as_float((uint32_t)(e2 + 127) << 23);
#pragma unroll
    for (int d = 0; d < DPL; ++d) q_s[gg * HD + lane * DPL + d] = qr[d] * sc;
    if (lane == 0) qs_s[gg] = __uint_as_float((uint32_t)(127 - e2) << 23);
  }
  if (owns_new) {
    float kx[DPL], vx[DPL];
    const float* kp = qrow + (a.nq + h) * HD + lane * DPL;
    const float* vp = qrow + (a.nq + a.nkv + h) * HD + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      kx[d] = kp[d];
      vx[d] = vp[d];
    }
    norm_rope_head<HD, DPL>(kx, gk, a.eps, cs, sn, lane, rope_ok, a.gk != nullptr);
    __half* kd = cache_row<__half, HD>(const_cast<void*>(a.kc), seq_ok ? seq : -1, h, new_slot, a.cache);
    __half* vd = cache_row<__half, HD>(const_cast<void*>(a.vc), seq_ok ? seq : -1, h, new_slot, a.cache);
    if (kd != nullptr && vd != nullptr) {
#pragma unroll
      for (int d = 0; d < DPL; ++d) {
        kd[lane * DPL + d] = __float2half_rn(kx[d]);
        vd[lane * DPL + d] = __float2half_rn(vx[d]);
      }
    } else if (lane == 0) {
      set_status(a.status, TQ_DEV_KV_OVERFLOW);
    }
    __threadfence();
    fence_proxy_async_global();  // the new row is read back by this warp's tensor copies
    __syncwarp();
    if (my_n == 1) stage(0);
  }
  __syncthreads();  // q_s, qs_s

  // B fragments of the query group: column 2j + part of n-tile nt is head 4 nt + j
  uint32_t qb[NT][KS][2];
  float inv_q[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 4 + (g >> 1);
    const bool lo = (g & 1) != 0;
    inv_q[nt] = (nt * 4 + c) < G ? qs_s[nt * 4 + c] : 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (hh < G) {
        const float* qv = q_s + hh * HD + ks * 16 + 2 * c;
        qb[nt][ks][0] = split_pair(qv[0], qv[1], lo);
        qb[nt][ks][1] = split_pair(qv[8], qv[9], lo);
      } else {
        qb[nt][ks][0] = qb[nt][ks][1] = 0u;
      }
    }
  }

  float m_run[NT], l_run[NT], o[NT][KS][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = kNegInf;
    l_run[nt] = 0.f;
#pragma unroll
    for (int md = 0; md < KS; ++md) o[nt][md][0] = o[nt][md][1] = o[nt][md][2] = o[nt][md][3] = 0.f;
  }
  // copies in flight at the top of iteration k: K(k), V(k)
  for (int k = 0; k < my_n; ++k) {
    wait_tile(k, false);  // K(k): rows past the context only meet masked scores
    zero_rows(kt, k);     // (a page outside the pool: zeros, as for V)
    const int nv = min(TILE, k1 - tile_key0(k));
    const int nlo = lo - tile_key0(k);  // keys of the tile before the window
    // scores of the tile: two m-tiles of 16 keys
    float sc[NT][2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sc[nt][mt][0] = sc[nt][mt][1] = sc[nt][mt][2] = sc[nt][mt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int key = mt * 16 + (lane & 15), ch = 2 * ks + (lane >> 4);
        uint32_t af[4];
        ldsm_x4(tile_chunk(kt_s, key, ch), af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16(sc[nt][mt], af, qb[nt][ks][0], qb[nt][ks][1]);
      }
    }
    __syncwarp();  // every lane is done with K(k): load K(k+1) behind the rest of this tile
    if (k + 1 < my_n) stage_one(k + 1, false);
    // online softmax per head (this thread: head 4 nt + c, keys g, g+8, 16+g, 24+g)
    float alpha[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float s4[4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int ka = mt * 16 + g, kb = ka + 8;
        s4[2 * mt] = ka < nv && ka >= nlo ? (sc[nt][mt][0] + sc[nt][mt][1]) * inv_q[nt] : kNegInf;
        s4[2 * mt + 1] = kb < nv && kb >= nlo ? (sc[nt][mt][2] + sc[nt][mt][3]) * inv_q[nt] : kNegInf;
      }
      float mt_ = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
      mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, 4));
      mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, 8));
      mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, 16));
      const float m_new = fmaxf(m_run[nt], mt_);
      alpha[nt] = m_run[nt] == kNegInf ? 0.f : exp2f(m_run[nt] - m_new);
      float ps = 0.f;
      const int hh = nt * 4 + c;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = m_new == kNegInf ? 0.f : exp2f(s4[i] - m_new);
        ps += p;
        if (hh < G) p_s[hh * 32 + (i >> 1) * 16 + g + (i & 1) * 8] = p;
      }
      ps += __shfl_xor_sync(0xffffffffu, ps, 4);
      ps += __shfl_xor_sync(0xffffffffu, ps, 8);
      ps += __shfl_xor_sync(0xffffffffu, ps, 16);
      l_run[nt] = l_run[nt] * alpha[nt] + ps;
      m_run[nt] = m_new;
#pragma unroll
      for (int md = 0; md < KS; ++md)
#pragma unroll
        for (int r = 0; r < 4; ++r) o[nt][md][r] *= alpha[nt];
    }
    wait_tile(k, true);  // V(k)
    zero_rows(vt, k);
    // O^T += V^T P^T: two k-steps of 16 keys
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int hh = nt * 4 + (g >> 1);
        const bool lo = (g & 1) != 0;
        if (hh < G) {
          const float* pv = p_s + hh * 32 + kk * 16 + 2 * c;
          pb[nt][0] = split_pair(pv[0] * 16384.f, pv[1] * 16384.f, lo);
          pb[nt][1] = split_pair(pv[8] * 16384.f, pv[9] * 16384.f, lo);
        } else {
          pb[nt][0] = pb[nt][1] = 0u;
        }
      }
#pragma unroll
      for (int md = 0; md < KS; ++md) {
        const int mi = lane >> 3;
        const int key = kk * 16 + (lane & 7) + ((mi >> 1) & 1) * 8, ch = 2 * md + (mi & 1);
        uint32_t af[4];
        ldsm_x4_t(tile_chunk(vt_s, key, ch), af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16(o[nt][md], af, pb[nt][0], pb[nt][1]);
      }
    }
    __syncwarp();  // p_s and the V buffer are rewritten next
    if (k + 1 < my_n) stage_one(k + 1, true);
  }
  // after a wait gave up (no copy was issued after it), the copy it waited
  // for lands before the CTA exits
  if (pend_k >= 0) mbar_wait_timed(kbar, (uint32_t)pend_k, kTileWaitNs);
  if (pend_v >= 0) mbar_wait_timed(vbar, (uint32_t)pend_v, kTileWaitNs);

  // ---- this warp's (m, l, o) per head into shared memory, then merge as the
  // scalar path does
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 4 + c;
    if (hh < G) {
      if (g == 0) {
        m_s[warp * G + hh] = m_run[nt];
        l_s[warp * G + hh] = l_run[nt];
      }
#pragma unroll
      for (int md = 0; md < KS; ++md) {
        o_s[(warp * G + hh) * HD + md * 16 + g] = (o[nt][md][0] + o[nt][md][1]) * (1.0f / 16384.f);
        o_s[(warp * G + hh) * HD + md * 16 + g + 8] = (o[nt][md][2] + o[nt][md][3]) * (1.0f / 16384.f);
      }
    }
  }
  __syncthreads();
  float* res_m = reinterpret_cast<float*>(smem + S::OFF_RES);
  float* res_l = res_m + G;
  float* res_o = res_l + G;
  for (int i = tid; i < G * HD; i += 128) {
    const int gg = i / HD, d = i % HD;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, m_s[w * G + gg]);
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = M == kNegInf ? 0.f : exp2f(m_s[w * G + gg] - M);
      acc += f * o_s[(w * G + gg) * HD + d];
      L += f * l_s[w * G + gg];
    }
    res_o[i] = acc;
    if (d == 0) {
      res_m[gg] = M;
      res_l[gg] = L;
    }
  }
  // push: rank q finishes outputs [q SHARE, (q+1) SHARE); every rank writes
  // its partial of that range and its (m, l) into rank q's inbox, then one
  // cluster barrier, then each rank merges from its own shared memory
  constexpr int SHARE = S::SHARE;
  constexpr int ROW = SHARE + 2 * G;
  float* inbox = reinterpret_cast<float*>(smem + S::OFF_IN);
  __syncthreads();  // res_* complete
  for (int i = tid; i < CL * ROW; i += 128) {
    const int q = i / ROW, j = i % ROW;
    const float v = j < SHARE ? res_o[q * SHARE + j] : j < SHARE + G ? res_m[j - SHARE] : res_l[j - SHARE - G];
    st_cluster_f32(map_cluster(inbox + split * ROW + j, q), v);
  }
  cluster_sync_all();
  for (int i = tid; i < SHARE; i += 128) {
    const int o_idx = split * SHARE + i, gg = o_idx / HD;
    float M = kNegInf;
#pragma unroll
    for (int r = 0; r < CL; ++r) M = fmaxf(M, inbox[r * ROW + SHARE + gg]);
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int r = 0; r < CL; ++r) {
      const float mr = inbox[r * ROW + SHARE + gg];
      const float f = mr == kNegInf ? 0.f : exp2f(mr - M);
      acc += f * inbox[r * ROW + i];
      L += f * inbox[r * ROW + SHARE + G + gg];
    }
    a.o[(int64_t)t * a.nq * HD + (h * G) * HD + o_idx] = acc / L;
  }
}

template <int HD, int G, int CL, bool FUSED>
cudaError_t attn_tc_cl(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a, cudaStream_t s) {
  using S = TcSmem<HD, G, CL>;
  static PerDevice setup;
  cudaError_t e = per_device(setup, nullptr, [](int, int&) {
    cudaError_t r = cudaFuncSetAttribute(attn_tc_kernel<HD, G, CL, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
    if (r == cudaSuccess && CL > 8)
      r = cudaFuncSetAttribute(attn_tc_kernel<HD, G, CL, FUSED>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return r;
  });
  if (e != cudaSuccess) return e;
  return launch_cluster(attn_tc_kernel<HD, G, CL, FUSED>, dim3(CL, a.nkv, a.T), dim3(128), S::BYTES, CL, s, kmap, vmap,
                        a);
}

// One token: 16 CTAs per KV head share its context (parallelism for one
// sequence).  Several tokens (batched decode): 4 CTAs per (token, KV head),
// so every warp has several tiles to pipeline and the launch still has
// thousands of CTAs.
template <int HD, int G>
cudaError_t attn_tc_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a, cudaStream_t s) {
  return a.T == 1 ? attn_tc_cl<HD, G, kCluster, true>(kmap, vmap, a, s) : attn_tc_cl<HD, G, 4, true>(kmap, vmap, a, s);
}

template <typename KT, int HD>
cudaError_t rope_t(const RopeArgs& a, cudaStream_t s) {
  dim3 grid((a.nq + a.nkv + 3) / 4, a.T);
  return launch_k(rope_append_kernel<KT, HD>, grid, dim3(128), 0, s, a);
}

template <typename KT, int HD, int G, int NS>
cudaError_t attn_configure() {
  using S = AttnSmem<KT, HD, G, NS>;
  static PerDevice setup;
  return per_device(setup, nullptr, [](int, int&) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<KT, HD, G, NS, false, 0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_decode_kernel<KT, HD, G, NS, true, kCluster>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_decode_kernel<KT, HD, G, NS, true, kCluster>,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
}

template <typename KT, int HD, int G, int NS>
cudaError_t attn_t(const AttnArgs& a, cudaStream_t s) {
  using S = AttnSmem<KT, HD, G, NS>;
  cudaError_t e = attn_configure<KT, HD, G, NS>();
  if (e != cudaSuccess) return e;
  if (!a.fused) {
    dim3 grid(a.max_splits, a.nkv, a.T);
    return launch_k(attn_decode_kernel<KT, HD, G, NS, false, 0>, grid, dim3(128), S::BYTES, s, a);
  }
  // decode: one cluster of kCluster CTAs per (token, KV head)
  return launch_cluster(attn_decode_kernel<KT, HD, G, NS, true, kCluster>, dim3(kCluster, a.nkv, a.T),
                        dim3(128), S::BYTES, kCluster, s, a);
}

// Decode (clusters of kCluster CTAs): one stage per warp, so a CTA takes
// about a third of an SM's shared memory and every cluster of the launch
// finds room at once (with two stages only part of the clusters fit, and
// the rest ran as a second wave).  Prefill: two stages when a warp may have
// several tiles, except for f32 rows of 128 dimensions (the second stage
// would not fit in shared memory).
template <typename KT, int HD, int G>
cudaError_t attn_g(const CUtensorMap* kmap, const CUtensorMap* vmap, const AttnArgs& a, cudaStream_t s) {
  if (sizeof(KT) == 2) {
    if (kmap == nullptr || vmap == nullptr) return cudaErrorInvalidValue;  // f16 caches are staged by TMA
    if (a.fused) return attn_tc_t<HD, G>(*kmap, *vmap, a, s);
    // rows of a mixed step (those not in a flash block: decode tokens, the
    // ragged ends of prompt chunks): 4 CTAs per (row, KV head) share the row's
    // causal prefix, as in batched decode
    return attn_tc_cl<HD, G, 4, false>(*kmap, *vmap, a, s);
  }
  if (a.fused || a.split_keys <= 4 * 32 || (sizeof(KT) == 4 && HD == 128)) return attn_t<KT, HD, G, 1>(a, s);
  return attn_t<KT, HD, G, 2>(a, s);
}

template <typename KT, int HD>
cudaError_t attn_h(int G, const CUtensorMap* kmap, const CUtensorMap* vmap, const AttnArgs& a, cudaStream_t s) {
  switch (G) {
    case 1: return attn_g<KT, HD, 1>(kmap, vmap, a, s);
    case 2: return attn_g<KT, HD, 2>(kmap, vmap, a, s);
    case 4: return attn_g<KT, HD, 4>(kmap, vmap, a, s);
    case 8: return attn_g<KT, HD, 8>(kmap, vmap, a, s);
  }
  return cudaErrorInvalidValue;
}

template <typename KT, int HD, int G>
cudaError_t prep_g() {
  cudaError_t e = attn_configure<KT, HD, G, 1>();
  if (e == cudaSuccess && !(sizeof(KT) == 4 && HD == 128)) e = attn_configure<KT, HD, G, 2>();
  return e;
}

template <typename KT, int HD>
cudaError_t prep_h(int G) {
  switch (G) {
    case 1: return prep_g<KT, HD, 1>();
    case 2: return prep_g<KT, HD, 2>();
    case 4: return prep_g<KT, HD, 4>();
    case 8: return prep_g<KT, HD, 8>();
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t attn_prepare(int kvtype, int hd, int G) {
  if (kvtype == TQ_KV_F16) return hd == 128 ? prep_h<__half, 128>(G) : prep_h<__half, 64>(G);
  return hd == 128 ? prep_h<float, 128>(G) : prep_h<float, 64>(G);
}

cudaError_t launch_rope_append(int kvtype, int hd, const RopeArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (kvtype == TQ_KV_F16) return hd == 128 ? rope_t<__half, 128>(a, s) : rope_t<__half, 64>(a, s);
  return hd == 128 ? rope_t<float, 128>(a, s) : rope_t<float, 64>(a, s);
}

cudaError_t launch_attn_decode(int kvtype, int hd, int G, const CUtensorMap* kmap, const CUtensorMap* vmap,
                               const AttnArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (kvtype == TQ_KV_F16)
    return hd == 128 ? attn_h<__half, 128>(G, kmap, vmap, a, s) : attn_h<__half, 64>(G, kmap, vmap, a, s);
  return hd == 128 ? attn_h<float, 128>(G, kmap, vmap, a, s) : attn_h<float, 64>(G, kmap, vmap, a, s);
}

}  // namespace tq
