// Temperature / top-p sampling on the device ("Всередині LLM: чисте виконання
// на Python для Qwen3-0.6B на MLX", step 8, sample(logits, temperature,
// top_p)): temperature 0 is the argmax (lowest index on ties); otherwise the
// tempered softmax's tokens in descending order of probability (ties by
// ascending index), the smallest prefix whose cumulative probability reaches
// top_p kept and renormalised, and the draw is the first kept token whose
// cumulative probability exceeds u (a uniform number the caller supplies).
//
// Masses.  Token i's unnormalised mass is the f32 exp2(-d_i), d_i = (max -
// l_i) log2(e) / T, held as an integer multiple of 2^-F with F = 62 -
// ceil(log2 V), so that V masses of at most 1 sum below 2^62.  Integer sums
// are exact in any order, so the draw does not depend on timing, and the
// rounding (at most 2^-F-1 per token, V 2^-F-1 <= 2^-25 of the total mass)
// lies far below the f32 exp's own.  Both targets become integers: the cutoff
// is the first token whose inclusive cumulative mass reaches ceil(top_p Z),
// the draw the first whose cumulative mass reaches floor(u kept) + 1.  A
// token whose mass rounds to 0 is never the first to reach a target >= 1 and
// is skipped everywhere.
//
// One thread-block cluster per row (up to 16 CTAs at batch 1, fewer as the
// batch fills the GPU), each CTA over its own slice of the row; no sort of
// the row:
//  1. the row's largest logit (each rank's maximum pushed to every rank);
//  2. a histogram of masses and counts over 2048 bins of d (32 per halving of
//     the mass): each bin is a contiguous run of the descending order, and
//     the tokens spread over many bins, so the shared-memory atomics seldom
//     meet (a radix histogram over the logits' leading bits puts nearly every
//     token in two or three bins);
//     each rank bins its slice, then sums one share of the bins over all
//     ranks (distributed shared memory) into rank 0;
//  3. on rank 0, a prefix sum over the bins finds the bin in which the
//     cumulative mass reaches the cutoff; every rank appends that bin's tokens
//     of its slice to rank 0's list, which rank 0 sorts by (logit descending,
//     index ascending) and sums in that order: the cutoff token and the kept
//     mass, exactly;
//  4. the same for the draw (the sorted bin is reused when the draw falls in
//     it).
// Every rank passes the same seven cluster barriers; what the ranks do
// between them is decided on rank 0 and pushed to every rank first.
// A bin of more than kCap tokens is resolved on rank 0 alone by a radix select
// over the bin's logit keys, then over the indices of the tie group that holds
// the target, with warp-aggregated counts.  The row is read once per pass (three
// or four passes in the common case), each thread with four 16-byte loads in
// flight.
#include <cooperative_groups.h>
#include <cooperative_groups/reduce.h>

#include "kernels.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace tq {
namespace smp {

namespace cg = cooperative_groups;

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;      // bins of d, 32 per halving of the mass
constexpr int kCap = 4096;       // tokens of one bin sorted in shared memory
constexpr int kNone = 256;       // "no digit" label of the radix fallback
constexpr int kMaxCluster = 16;  // CTAs per row at most
typedef unsigned long long u64;

struct Smem {
  u64 cum[kBins];        // bin masses, then their inclusive prefix sums
  unsigned cnt[kBins];   // tokens of nonzero mass per bin
  u64 list[kCap];        // gathered tokens: (~key << 32) | index, sorted ascending
  u64 lcum[kCap];        // inclusive prefix sums of the sorted tokens' masses
  u64 dmass[256];        // radix fallback: mass and count per digit
  unsigned dcnt[256];
  u64 wsum[kWarps];
  unsigned long long best[kWarps];
  float fred[kWarps];
  int n_list, found;
  u64 found_cum;
  unsigned prefix;
  u64 above;
  // cluster: rank 0's merged histogram, and what each rank receives
  u64 mcum[kBins];       // merged bin masses, then their inclusive prefix sums
  unsigned mcnt[kBins];
  float fin[kMaxCluster];             // every rank's largest logit
  unsigned long long kin[kMaxCluster];  // every rank's argmax key (greedy)
  int ctl_bin, ctl_mode;              // the cutoff bin; 0: gather it, 1: rank 0 alone
  int ctl2_bin, ctl2_need;            // the draw bin; 1: gather it
};

// d -> bin: d * 32 rounded to an integer through the f32 mantissa (monotone
// in d, the same in every pass), at most kBins - 1.
__device__ __forceinline__ int bin_of(float d) {
  const float x = fminf(d * 32.f, (float)(kBins - 1));
  return (int)(__float_as_uint(x + 8388608.f) - 0x4B000000u);
}

// exp2(-d) as an integer multiple of 2^-F, rounded to nearest (half up), from
// the f32 bits: m = (2^23 + mantissa) 2^(e - 150).
__device__ __forceinline__ u64 mass_fix(float d, int F) {
  if (!(d < 126.f)) return 0ull;  // also NaN
  const uint32_t b = __float_as_uint(exp2f(-d));
  const int e = (int)(b >> 23);
  if (e == 0) return 0ull;
  const u64 m = (u64)((b & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 150 + F;
  if (sh >= 0) return m << sh;
  if (sh < -24) return 0ull;
  return (m + (1ull << (-sh - 1))) >> (-sh);
}

// Calls fn(i, l, ok) for every token i in [lo, hi) of the row, warp-uniformly
// (every thread makes the same number of calls; ok is false for padding),
// with kU float4 loads of each thread in flight before any is used (a pass is
// bound by load latency otherwise).  lo is a multiple of 4; rows that are not
// 16-byte aligned are read as scalars, kU * 4 at a time.
constexpr int kU = 4;
template <typename Fn>
__device__ __forceinline__ void walk_row(const float* row, int lo, int hi, Fn&& fn) {
  const int tid = threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0u) {
    const int j_lo = lo >> 2, j_hi = hi >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    for (int j0 = j_lo; j0 < j_hi; j0 += kThreads * kU) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u * kThreads + tid;
        v[u] = j < j_hi ? __ldg(r4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // four copies of fn per pass, not 4 kU (the kernel's hot code then stays
      // in the instruction cache); v[u] is picked by predicated moves, so
      // the loads stay in registers
#pragma unroll 1
      for (int u = 0; u < kU; ++u) {
        float4 c = v[0];
#pragma unroll
        for (int w = 1; w < kU; ++w)
          if (u == w) c = v[w];
        const int j = j0 + u * kThreads + tid;
        const bool ok = j < j_hi;
        fn(4 * j, c.x, ok);
        fn(4 * j + 1, c.y, ok);
        fn(4 * j + 2, c.z, ok);
        fn(4 * j + 3, c.w, ok);
      }
    }
    const int i = 4 * j_hi + tid;  // hi % 4 tokens past the last whole float4
    fn(i, i < hi ? __ldg(row + i) : 0.f, i < hi);
  } else {
    for (int i0 = lo; i0 < hi; i0 += kThreads * 4 * kU) {
      float v[4 * kU];
#pragma unroll
      for (int u = 0; u < 4 * kU; ++u) {
        const int i = i0 + u * kThreads + tid;
        v[u] = i < hi ? __ldg(row + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4 * kU; ++u) {
        const int i = i0 + u * kThreads + tid;
        fn(i, v[u], i < hi);
      }
    }
  }
}

// Inclusive prefix sum in place of a[0 .. PER * kThreads) (entries >= n read
// as 0 and left alone); every thread of the CTA calls it.
template <int PER>
__device__ void block_scan(u64* a, int n, u64* wsum) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  u64 v[PER];
  u64 s = 0ull;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = t * PER + k;
    s += i < n ? a[i] : 0ull;
    v[k] = s;
  }
  u64 x = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const u64 y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    u64 z = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const u64 y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    wsum[lane] = z;
  }
  __syncthreads();
  const u64 off = (w > 0 ? wsum[w - 1] : 0ull) + (x - s);
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = t * PER + k;
    if (i < n) a[i] = v[k] + off;
  }
  __syncthreads();
}

// The bin in which the inclusive cumulative mass (prefix sums `cum`) first
// reaches T (1 <= T <= Z).
__device__ int find_bin(Smem& sm, const u64* cum, u64 T) {
  if (threadIdx.x == 0) sm.found = kBins - 1;
  __syncthreads();
  for (int b = threadIdx.x; b < kBins; b += kThreads) {
    const u64 lo = b > 0 ? cum[b - 1] : 0ull;
    if (lo < T && T <= cum[b]) sm.found = b;  // at most one bin qualifies
  }
  __syncthreads();
  const int r = sm.found;
  __syncthreads();
  return r;
}

struct Pick {
  int index;
  u64 cum;  // inclusive cumulative mass at the picked token
};

// Append the tokens of bin `bin` in [lo, hi) of the row to dst's list (this
// CTA's shared memory or rank 0's, through the cluster window): one atomic
// per warp reserves the warp's slots.
__device__ void gather(Smem* dst, const float* row, int lo, int hi, float lmax, float sc, int F, int bin) {
  const int lane = threadIdx.x & 31;
  walk_row(row, lo, hi, [&](int i, float l, bool ok) {
    bool hit = false;
    if (ok) {
      const float d = (lmax - l) * sc;
      hit = bin_of(d) == bin && mass_fix(d, F) != 0ull;
    }
    const unsigned ball = __ballot_sync(0xffffffffu, hit);
    if (ball != 0u) {
      const int leader = __ffs(ball) - 1;
      int base = 0;
      if (lane == leader) base = atomicAdd(&dst->n_list, __popc(ball));
      base = __shfl_sync(0xffffffffu, base, leader);
      const int at = base + __popc(ball & ((1u << lane) - 1u));
      if (hit && at < kCap) dst->list[at] = ((u64)(~float_order_key(l)) << 32) | (u64)(uint32_t)i;
    }
  });
}

// Sort this CTA's list of n <= kCap gathered tokens by (logit descending,
// index ascending) and prefix-sum their masses.
__device__ void sort_scan(Smem& sm, const float* row, float lmax, float sc, int F, int n) {
  const int tid = threadIdx.x;
  int m = 2;
  while (m < n) m <<= 1;
  for (int i = n + tid; i < m; i += kThreads) sm.list[i] = ~0ull;
  __syncthreads();
  if (m <= kThreads) {
    // one element per thread: exchanges at distance < 32 by warp shuffles,
    // the others through shared memory (a pair (i, i ^ j) keeps its smaller
    // key at i in an ascending run, at i ^ j in a descending one)
    u64 v = tid < m ? sm.list[tid] : ~0ull;
    for (int k = 2; k <= m; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        u64 o;
        if (j >= 32) {
          if (tid < m) sm.list[tid] = v;
          __syncthreads();
          o = tid < m ? sm.list[tid ^ j] : v;
          __syncthreads();
        } else {
          o = __shfl_xor_sync(0xffffffffu, v, j);
        }
        const bool keep_min = ((tid & j) == 0) == ((tid & k) == 0);
        v = keep_min ? (o < v ? o : v) : (o > v ? o : v);
      }
    }
    if (tid < m) sm.list[tid] = v;
    __syncthreads();
  } else {
    for (int k = 2; k <= m; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int t = tid; t < m / 2; t += kThreads) {
          const int i = (t / j) * 2 * j + (t % j), p = i + j;
          const u64 a = sm.list[i], b = sm.list[p];
          if ((a > b) == ((i & k) == 0)) {
            sm.list[i] = b;
            sm.list[p] = a;
          }
        }
        __syncthreads();
      }
    }
  }
  for (int i = tid; i < n; i += kThreads) {
    const int idx = (int)(uint32_t)(sm.list[i] & 0xFFFFFFFFull);
    sm.lcum[i] = mass_fix((lmax - __ldg(row + idx)) * sc, F);
  }
  __syncthreads();
  block_scan<kCap / kThreads>(sm.lcum, n, sm.wsum);
}

// Radix fallback for a bin too large to sort: the key (8 bits a level, top
// down; larger digits come first in the order), then the r-th lowest index
// among the tokens of that key.  Counts and masses per digit are summed over
// each warp's lanes of equal digit before one shared-memory atomic.
__device__ __noinline__ Pick radix_pick(Smem& sm, const float* row, int V, float lmax, float sc, int F, int bin,
                                        u64 base, u64 T) {
  const int tid = threadIdx.x;
  auto warp = cg::tiled_partition<32>(cg::this_thread_block());
  if (tid == 0) {
    sm.prefix = 0u;
    sm.above = base;
  }
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int k = tid; k < 256; k += kThreads) {
      sm.dmass[k] = 0ull;
      sm.dcnt[k] = 0u;
    }
    __syncthreads();
    const uint32_t prefix = sm.prefix;
    walk_row(row, 0, V, [&](int i, float l, bool ok) {
      int dg = kNone;
      u64 mf = 0ull;
      if (ok) {
        const float d = (lmax - l) * sc;
        const uint32_t key = float_order_key(l);
        if (bin_of(d) == bin && (shift == 24 || (key >> (shift + 8)) == (prefix >> (shift + 8)))) {
          mf = mass_fix(d, F);
          if (mf != 0ull) dg = (int)((key >> shift) & 255u);
        }
      }
      if (__any_sync(0xffffffffu, dg != kNone)) {
        auto g = cg::labeled_partition(warp, dg);
        const u64 s = cg::reduce(g, mf, cg::plus<u64>());
        if (g.thread_rank() == 0 && dg != kNone) {
          atomicAdd(&sm.dmass[dg], s);
          atomicAdd(&sm.dcnt[dg], (unsigned)g.size());
        }
      }
    });
    __syncthreads();
    if (tid == 0) {
      u64 cum = sm.above;
      int chosen = -1, last = -1;
      u64 cum_last = cum;
      for (int k = 255; k >= 0; --k) {
        if (sm.dcnt[k] == 0u) continue;
        if (cum + sm.dmass[k] >= T) {
          chosen = k;
          break;
        }
        last = k;
        cum_last = cum;
        cum += sm.dmass[k];
      }
      if (chosen < 0) {  // not reached inside the bin (cannot happen for a T inside it): its last group
        chosen = last < 0 ? 0 : last;
        cum = cum_last;
      }
      sm.above = cum;
      sm.prefix = prefix | ((uint32_t)chosen << shift);
    }
    __syncthreads();
  }
  // the tie group of key K: n tokens of one mass m1 each, `above` before them
  const uint32_t K = sm.prefix;
  const u64 above = sm.above;
  const unsigned n_tie = sm.dcnt[K & 255u];
  const u64 m_tie = sm.dmass[K & 255u];
  __syncthreads();
  const u64 m1 = n_tie > 0u ? m_tie / n_tie : 1ull;
  u64 r = T > above ? (T - above + m1 - 1ull) / m1 : 1ull;  // tokens of the group needed
  if (r < 1ull) r = 1ull;
  if (r > n_tie) r = n_tie > 0u ? n_tie : 1u;
  // the r-th lowest index among the tokens of key K
  if (tid == 0) {
    sm.prefix = 0u;
    sm.found_cum = 0ull;  // tokens before the chosen index digits
  }
  for (int shift = 16; shift >= 0; shift -= 8) {
    for (int k = tid; k < 256; k += kThreads) sm.dcnt[k] = 0u;
    __syncthreads();
    const uint32_t prefix = sm.prefix;
    walk_row(row, 0, V, [&](int i, float l, bool ok) {
      int dg = kNone;
      if (ok && float_order_key(l) == K &&
          (shift == 16 || ((uint32_t)i >> (shift + 8)) == (prefix >> (shift + 8))))
        dg = (int)(((uint32_t)i >> shift) & 255u);
      if (__any_sync(0xffffffffu, dg != kNone)) {
        auto g = cg::labeled_partition(warp, dg);
        if (g.thread_rank() == 0 && dg != kNone) atomicAdd(&sm.dcnt[dg], (unsigned)g.size());
      }
    });
    __syncthreads();
    if (tid == 0) {
      u64 before = sm.found_cum;
      int chosen = 255;
      for (int k = 0; k < 256; ++k) {  // ascending index
        if (before + sm.dcnt[k] >= r) {
          chosen = k;
          break;
        }
        before += sm.dcnt[k];
      }
      sm.found_cum = before;
      sm.prefix = prefix | ((uint32_t)chosen << shift);
    }
    __syncthreads();
  }
  Pick p;
  p.index = (int)sm.prefix;
  p.cum = above + r * m1;
  __syncthreads();
  return p;
}

// The first token of the sorted list (n tokens of one bin, `base` the mass
// before the bin) whose inclusive cumulative mass reaches T.
__device__ Pick pick_list(Smem& sm, int n, u64 base, u64 T) {
  if (threadIdx.x == 0) {
    sm.found = n - 1;
    sm.found_cum = base + (n > 0 ? sm.lcum[n - 1] : 0ull);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const u64 lo = base + (i > 0 ? sm.lcum[i - 1] : 0ull);
    const u64 hi = base + sm.lcum[i];
    if (lo < T && T <= hi) {  // exactly one position
      sm.found = i;
      sm.found_cum = hi;
    }
  }
  __syncthreads();
  Pick p;
  p.index = n > 0 ? (int)(uint32_t)(sm.list[sm.found] & 0xFFFFFFFFull) : -1;
  p.cum = sm.found_cum;
  __syncthreads();
  return p;
}

template <int CL>
__global__ void __launch_bounds__(kThreads, 1) sample_kernel(const float* logits, int V, const float* temperature,
                                                              const float* top_p, const float* u, int32_t* out) {
  // every CTA of the cluster has started before any of them touches another's
  // shared memory: arrive here, wait before the first remote store
  cluster_arrive_relaxed();
  grid_dep_launch();
  grid_dep_wait();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  Smem* s0 = cluster.map_shared_rank(&sm, 0u);  // rank 0's shared memory
  const int b = blockIdx.y, tid = threadIdx.x;
  const float* row = logits + (int64_t)b * V;
  // this rank's slice: whole float4 groups, the last rank also takes the tail
  const int G4 = V >> 2;
  const int i_lo = 4 * (int)((int64_t)G4 * rank / CL);
  const int i_hi = rank == CL - 1 ? V : 4 * (int)((int64_t)G4 * (rank + 1) / CL);
  const float T = temperature[b];

  // 1. the largest logit, pushed to every rank
  float mx = -3.402823466e38f;
  walk_row(row, i_lo, i_hi, [&](int, float l, bool ok) {
    if (ok) mx = fmaxf(mx, l);
  });
  mx = warp_max(mx);
  if ((tid & 31) == 0) sm.fred[tid >> 5] = mx;
  __syncthreads();
  cluster_wait();
  if (tid < CL) {
    float m = sm.fred[0];
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, sm.fred[w]);
    cluster.map_shared_rank(&sm, (unsigned)tid)->fin[rank] = m;
  }
  cluster.sync();  // barrier 1
  float lmax = sm.fin[0];
  for (int r = 1; r < CL; ++r) lmax = fmaxf(lmax, sm.fin[r]);

  if (!(T > 0.f) || !(lmax <= 3.402823466e38f)) {
    // greedy (also for a row whose largest logit is +inf): lowest index of the largest logit
    unsigned long long best = 0ull;
    walk_row(row, i_lo, i_hi, [&](int i, float l, bool ok) {
      const unsigned long long k = ok ? argmax_key(l, (uint32_t)i) : 0ull;
      best = k > best ? k : best;
    });
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    if ((tid & 31) == 0) sm.best[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = sm.best[0];
      for (int w = 1; w < kWarps; ++w) m = sm.best[w] > m ? sm.best[w] : m;
      s0->kin[rank] = m;
    }
    cluster.sync();  // the greedy path's only other barrier
    if (rank == 0 && tid == 0) {
      unsigned long long m = sm.kin[0];
      for (int r = 1; r < CL; ++r) m = sm.kin[r] > m ? sm.kin[r] : m;
      out[b] = (int32_t)argmax_key_index(m);
    }
    return;
  }
  const float sc = 1.4426950408889634f / T;  // log2(e) / T
  const int F = 62 - (V > 1 ? 32 - __clz(V - 1) : 0);

  // 2. this slice's histogram of masses and counts over the bins of d
  for (int k = tid; k < kBins; k += kThreads) {
    sm.cum[k] = 0ull;
    sm.cnt[k] = 0u;
  }
  if (tid == 0) sm.n_list = 0;
  __syncthreads();
  walk_row(row, i_lo, i_hi, [&](int, float l, bool ok) {
    const float d = (lmax - l) * sc;
    const u64 mf = ok ? mass_fix(d, F) : 0ull;
    if (mf != 0ull) {
      const int k = bin_of(d);
      atomicAdd(&sm.cum[k], mf);
      atomicAdd(&sm.cnt[k], 1u);
    }
  });
  cluster.sync();  // barrier 2: every slice's histogram is complete
  // this rank's share of the bins, summed over the ranks, into rank 0
  for (int k = kBins * rank / CL + tid; k < kBins * (rank + 1) / CL; k += kThreads) {
    u64 m = 0ull;
    unsigned c = 0u;
    for (int r = 0; r < CL; ++r) {
      const Smem* sr = cluster.map_shared_rank(&sm, (unsigned)r);
      m += sr->cum[k];
      c += sr->cnt[k];
    }
    s0->mcum[k] = m;
    s0->mcnt[k] = c;
  }
  cluster.sync();  // barrier 3: rank 0 holds the whole histogram

  // 3. the cutoff: the first token whose cumulative mass reaches ceil(top_p Z)
  Pick cut, draw;
  cut.index = draw.index = -1;
  cut.cum = draw.cum = 0ull;
  int c_bin = 0;
  u64 c_base = 0ull;
  if (rank == 0) {
    block_scan<kBins / kThreads>(sm.mcum, kBins, sm.wsum);
    const u64 Z = sm.mcum[kBins - 1];  // >= 2^F: the largest logit's mass is 1
    float tp = top_p[b];
    if (!(tp < 1.f)) tp = 1.f;  // also NaN
    if (!(tp > 0.f)) tp = 0.f;
    u64 Tc = (u64)ceil((double)tp * (double)Z);
    Tc = Tc < 1ull ? 1ull : Tc > Z ? Z : Tc;
    c_bin = find_bin(sm, sm.mcum, Tc);
    c_base = c_bin > 0 ? sm.mcum[c_bin - 1] : 0ull;
    if (tid == 0) {
      sm.found_cum = Tc;  // kept for rank 0's own use after the gather
      const int mode = sm.mcnt[c_bin] > (unsigned)kCap ? 1 : 0;
      for (int r = 0; r < CL; ++r) {
        Smem* sr = cluster.map_shared_rank(&sm, (unsigned)r);
        sr->ctl_bin = c_bin;
        sr->ctl_mode = mode;
      }
    }
  }
  cluster.sync();  // barrier 4: every rank knows the cutoff bin
  const int mode = sm.ctl_mode;
  if (mode == 0) gather(s0, row, i_lo, i_hi, lmax, sc, F, sm.ctl_bin);
  cluster.sync();  // barrier 5: rank 0's list holds the cutoff bin
  int need2 = 0;
  if (rank == 0) {
    const u64 Tc = sm.found_cum;
    if (mode == 0) {
      const int n = min(sm.n_list, kCap);
      sort_scan(sm, row, lmax, sc, F, n);
      cut = pick_list(sm, n, c_base, Tc);
    } else {
      cut = radix_pick(sm, row, V, lmax, sc, F, c_bin, c_base, Tc);
    }
    // 4. the draw: the first kept token whose cumulative mass exceeds u * kept
    float uu = u[b];
    if (!(uu > 0.f)) uu = 0.f;  // also NaN
    u64 Td = (u64)floor((double)uu * (double)cut.cum) + 1ull;
    Td = Td > cut.cum ? cut.cum : Td;
    const int d_bin = find_bin(sm, sm.mcum, Td);
    const u64 d_base = d_bin > 0 ? sm.mcum[d_bin - 1] : 0ull;
    if (d_bin == c_bin && mode == 0) {
      draw = pick_list(sm, min(sm.n_list, kCap), d_base, Td);
    } else if (sm.mcnt[d_bin] <= (unsigned)kCap) {
      need2 = 1;  // gathered by every rank
    } else {
      draw = radix_pick(sm, row, V, lmax, sc, F, d_bin, d_base, Td);
    }
    if (tid == 0) {
      sm.found_cum = Td;
      sm.n_list = 0;
      for (int r = 0; r < CL; ++r) {
        Smem* sr = cluster.map_shared_rank(&sm, (unsigned)r);
        sr->ctl2_bin = d_bin;
        sr->ctl2_need = need2;
      }
    }
  }
  cluster.sync();  // barrier 6: every rank knows whether to gather the draw bin
  if (sm.ctl2_need) gather(s0, row, i_lo, i_hi, lmax, sc, F, sm.ctl2_bin);
  cluster.sync();  // barrier 7: rank 0's list holds the draw bin; no remote access after this
  if (rank == 0) {
    if (sm.ctl2_need) {
      const int d_bin = sm.ctl2_bin;
      const int n = min(sm.n_list, kCap);
      sort_scan(sm, row, lmax, sc, F, n);
      draw = pick_list(sm, n, d_bin > 0 ? sm.mcum[d_bin - 1] : 0ull, sm.found_cum);
    }
    if (tid == 0) out[b] = draw.index >= 0 && draw.index < V ? draw.index
                           : cut.index >= 0 && cut.index < V ? cut.index : 0;
  }
}

}  // namespace smp

namespace {
template <int CL>
cudaError_t sample_setup() {
  cudaError_t e = cudaFuncSetAttribute(smp::sample_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(smp::Smem));
  if (e == cudaSuccess && CL > 8)
    e = cudaFuncSetAttribute(smp::sample_kernel<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

// Clusters of CL CTAs (one per SM) can be resident at once on this device.
template <int CL>
int sample_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, 1, 1);
  cfg.blockDim = dim3(smp::kThreads);
  cfg.dynamicSmemBytes = sizeof(smp::Smem);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = CL;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, smp::sample_kernel<CL>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int CL>
cudaError_t sample_launch(const float* logits, int batch, int V, const float* temperature, const float* top_p,
                          const float* u, int32_t* out, cudaStream_t s) {
  return launch_cluster(smp::sample_kernel<CL>, dim3(CL, batch, 1), dim3(smp::kThreads), sizeof(smp::Smem), CL, s,
                        logits, V, temperature, top_p, u, out);
}
}  // namespace

cudaError_t launch_sample(const float* logits, int batch, int V, const float* temperature, const float* top_p,
                          const float* u, int32_t* out, cudaStream_t s) {
  if (batch <= 0) return cudaSuccess;
  // the largest cluster the device runs, and the SM count
  static PerDevice setup;
  int caps = 0;
  cudaError_t e = per_device(setup, &caps, [](int dev, int& v) {
    cudaError_t r = sample_setup<1>();
    if (r == cudaSuccess) r = sample_setup<2>();
    if (r == cudaSuccess) r = sample_setup<4>();
    if (r == cudaSuccess) r = sample_setup<8>();
    if (r == cudaSuccess) r = sample_setup<16>();
    if (r != cudaSuccess) return r;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = kNumSMs;
    const int cl = sample_clusters<16>() > 0 ? 16 : sample_clusters<8>() > 0 ? 8 : sample_clusters<4>() > 0 ? 4
                   : sample_clusters<2>() > 0 ? 2 : 1;
    v = (sms << 8) | cl;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int sms = caps >> 8, cl_max = caps & 255;
  // rows x CTAs per row about the SM count: a row of one sequence gets up to 16 SMs
  int cl = 1;
  while (cl < cl_max && batch * cl * 2 <= sms) cl *= 2;
  switch (cl) {
    case 16: return sample_launch<16>(logits, batch, V, temperature, top_p, u, out, s);
    case 8: return sample_launch<8>(logits, batch, V, temperature, top_p, u, out, s);
    case 4: return sample_launch<4>(logits, batch, V, temperature, top_p, u, out, s);
    case 2: return sample_launch<2>(logits, batch, V, temperature, top_p, u, out, s);
  }
  return sample_launch<1>(logits, batch, V, temperature, top_p, u, out, s);
}

}  // namespace tq
