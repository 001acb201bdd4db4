// Internal launchers of the tq kernels (not part of the C ABI).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace tq {

// ---- tiled weight layout (tq_repack, the GEMV, decoding)
//
// Rows are grouped in tiles of 16 (a matrix's rows padded to a multiple of 16
// with zero rows) and the blocks of a tile row in units of 8 blocks (256
// inputs).  qs holds units [tile][unit] of 2048 (Q4_0) or 4096 (Q8_0) bytes,
// d holds units [tile][unit] of 128 fp16 scales; so a tile row is
// contiguous and a run of units is one contiguous copy.  Inside a unit, row
// rr = 8 h + g of the tile and word i (4 bytes; Q4_0 words 0-3, Q8_0 words
// 0-7) of block j (0-7) sit where one 16-byte load per lane of a warp hands
// lane 4 g + c the words its mma.m16n8k16 A fragment needs (c = i mod 4):
//   Q4_0: ((h*2 + j/4)*32 + 4g + i)*16 + (j%4)*4
//   Q8_0: ((h*4 + j/2)*32 + 4g + i%4)*16 + (j%2)*8 + (i/4)*4
// and the scale of (rr, j) is element (h*8 + g)*8 + j of the unit's scales.
constexpr int kTileRows = 16;
constexpr int kUnitBlocks = 8;
constexpr int kUnitD = 256;  // bytes of scales per unit

// 4-bit formats (Q4_0, AFFINE4) share the code arrangement; AFFINE4's
// scale elements hold (bf16 scale, bf16 bias) of each 64-input group.
__host__ __device__ constexpr bool nib4(int wt) { return wt != TQ_Q8_0; }
__host__ __device__ constexpr int unit_qs_bytes(int wt) { return nib4(wt) ? 2048 : 4096; }

__host__ __device__ inline int64_t tiled_rows(int64_t rows) { return (rows + 15) / 16 * 16; }

__host__ __device__ inline int64_t tiled_qs_offset(int wt, int64_t r, int64_t blk, int64_t nb, int i) {
  const int64_t unit = (r >> 4) * (nb / kUnitBlocks) + (blk >> 3);
  const int h = (int)((r >> 3) & 1), g = (int)(r & 7), j = (int)(blk & 7);
  if (nib4(wt)) return unit * 2048 + (int64_t)(((h * 2 + (j >> 2)) * 32 + g * 4 + i) * 16 + (j & 3) * 4);
  return unit * 4096 + (int64_t)(((h * 4 + (j >> 1)) * 32 + g * 4 + (i & 3)) * 16 + (j & 1) * 8 + (i >> 2) * 4);
}

__host__ __device__ inline int64_t tiled_d_index(int64_t r, int64_t blk, int64_t nb) {
  const int64_t unit = (r >> 4) * (nb / kUnitBlocks) + (blk >> 3);
  return unit * 128 + (((r >> 3) & 1) * 8 + (r & 7)) * 8 + (blk & 7);
}

// ---- block formats (quant.cu)
cudaError_t launch_quantize(int wtype, const float* w, int64_t n_blocks, void* out, cudaStream_t s);
cudaError_t launch_repack(int wtype, const void* src, int64_t rows, int64_t nb, void* qs,
                          uint16_t* d, cudaStream_t s);
cudaError_t launch_quantize_affine4(const float* w, int64_t rows, int64_t cols, uint32_t* words, uint16_t* scales,
                                    uint16_t* biases, cudaStream_t s);
cudaError_t launch_repack_affine4(const uint32_t* words, const uint16_t* scales, const uint16_t* biases,
                                  int64_t rows, int64_t cols, void* qs, uint16_t* d, cudaStream_t s);
cudaError_t launch_dequant(int wtype, const void* qs, const uint16_t* d, int64_t nb, int64_t row0,
                           int64_t n_rows, float* out, cudaStream_t s);
cudaError_t launch_embed(int wtype, const void* qs, const uint16_t* d, int vocab, int hidden,
                         const int32_t* tokens, int n_tokens, float* x, uint32_t* status,
                         unsigned long long* argmax_keys, int n_keys, cudaStream_t s);

// ---- decode GEMV (gemv.cu)
enum GemvMode { GEMV_STORE = 0, GEMV_SWIGLU = 1, GEMV_ARGMAX = 2 };
// activation of a gated FFN's gate: silu(z) = z / (1 + e^-z), or the tanh
// approximation of GELU, z/2 (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
enum GateAct { ACT_SILU = 0, ACT_GELU_TANH = 1 };

__device__ __forceinline__ float gate_act(float z, int act) {
  if (act == ACT_GELU_TANH) return 0.5f * z * (1.0f + tanhf(0.7978845608028654f * (z + 0.044715f * z * z * z)));
  return z / (1.0f + __expf(-z));
}

struct GemvSeg {
  const uint8_t* qs;
  const uint16_t* d;
  int rows;
};

struct GemvArgs {
  GemvSeg seg[3];        // STORE: row segments concatenated; SWIGLU: gate, up; ARGMAX: one
  int nseg;
  int K;                 // columns
  int N;                 // output rows (SWIGLU: ffn)
  int B;                 // tokens
  const float* x;        // [B][K]
  const float* gain;     // RMSNorm prologue gain [K], or null
  float eps;
  float* y;              // [B][N] (ARGMAX: logits, may be null)
  const float* residual; // [B][N] or null (STORE only); may alias y
  unsigned long long* argmax_keys;  // [B] (ARGMAX)
  uint32_t* status;      // device status word (bounded waits), or null
  const float* bias;     // STORE: [N] added to every output row, or null
  int act;               // SWIGLU: the gate's activation (ACT_SILU or ACT_GELU_TANH)
  float softcap;         // ARGMAX: logits = c tanh(logits / c) when c > 0
};

// Up to kMaxPhases GEMVs run by one persistent kernel; phase p+1 starts
// after every CTA finished phase p (grid-wide counters `sync`, [kMaxPhases+1]
// zeros between launches, which the kernel itself restores).
constexpr int kMaxPhases = 4;
constexpr int kMaxGrid = 256;  // CTAs of a GEMV launch at most
struct GemvChain {
  GemvArgs ph[kMaxPhases];
  int mode[kMaxPhases];
  int n;
  unsigned* sync;
  unsigned sync_limit;   // polls before a wait between phases gives up (0: the default)
};

// Returns cudaErrorInvalidValue when K has no supported thread mapping.
cudaError_t launch_gemv(int wtype, int mode, const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_chain(int wtype, const GemvChain& c, cudaStream_t s);
bool gemv_supported(int K);

// ---- tensor-core GEMM for prefill and batched decode (tcgemm.cu)
// Phase input rows -> fp16 rows after a power-of-two scale per row.
struct XPrep16Args {
  const float* x;
  const float* up;       // optional: the input is act(x) * up
  int act;               // GateAct of act()
  int ldx;
  const float* gain;     // optional RMSNorm gain
  float eps;
  int K, T;
  __half* x16;           // [T][K]
  float* inv_s;          // [T]: 2^-e of row t
};
// Y[t][r] (+)= sum_k W[r][k] X[t][k] over the concatenated segments, on tcgen05.
struct TcGemmArgs {
  GemvSeg seg[3];
  int nseg;
  int K, T;
  const __half* x16;       // [T][K], 16-byte aligned
  const float* inv_s;      // [T]
  float* y;                // [T][ldy]
  int ldy;
  const float* residual;   // [T][ldy] or null; may alias y
  const float* bias;       // [ldy] added to every row, or null
  uint32_t* status;
  // split over K (few token rows): part_cap floats of partial sums, n_counters
  // zero counters between launches; null part keeps one split
  float* part;
  int64_t part_cap;
  unsigned* counters;
  int n_counters;
};
cudaError_t launch_xprep16(const XPrep16Args& a, cudaStream_t s);
cudaError_t launch_tcgemm(int wtype, const TcGemmArgs& a, cudaStream_t s);

// ---- attention side (attn.cu)
struct CacheView {
  int max_ctx;               // slots per sequence (contiguous) or tokens per sequence (paged)
  int max_seq;               // sequences: cache slots (contiguous) or block-table rows (paged)
  int n_kv;
  int page_size;             // 0: contiguous [seq][n_kv][max_ctx][hd]; else pages [page][n_kv][page_size][hd]
  int n_pages;
  const int32_t* block_table;  // [seq][bt_stride]
  int bt_stride;
};

// Token t of a call belongs to sequence (seq_idx ? seq_idx[t] : seq_fixed >= 0
// ? seq_fixed : t), is rotated at position (pos ? pos[t] : pos_base + t) and
// stores / attends up to cache index (kv_len ? kv_len[t] : pos_base + t).
struct RopeArgs {
  float* qkv;                // [T][(nq + 2 nkv) * hd]: q rotated in place
  int T, nq, nkv;
  const int32_t* pos;
  const int32_t* kv_len;
  int pos_base;
  int seq_fixed;
  const int32_t* seq_idx;    // per-token sequence, or null
  void* kc;
  void* vc;                  // this layer's caches
  CacheView cache;
  const float* cos_t;        // [max_ctx][hd/2]
  const float* sin_t;
  const float* gq;           // per-head RMSNorm gains of q and k, or null: no norm
  const float* gk;
  float eps;
  uint32_t* status;
};

struct AttnArgs {
  const float* q;            // q of token t, head h: q + t*q_stride + h*hd
  int q_stride;
  float* o;                  // [T][nq*hd]
  int T, nq, nkv;
  const int32_t* kv_len;
  int pos_base;
  int seq_fixed;
  const int32_t* seq_idx;    // per-token sequence, or null
  const void* kc;
  const void* vc;
  CacheView cache;
  int split_keys;            // keys per split, a multiple of 32
  int max_splits;            // >= ceil(max_ctx / split_keys)
  float* part;               // [T][nkv][max_splits][G][hd + 2]
  unsigned* counters;        // [T][nkv], zero between calls
  float scale_log2;          // log2(e) / sqrt(hd)
  uint32_t* status;
  // fused decode: q, k, v come unnormalised from the Q/K/V projection (q points at
  // the [T][(nq + 2 nkv) hd] buffer); QK-RMSNorm, RoPE and the KV append happen here
  int fused;
  const int32_t* pos;        // rope position per token
  const float* cos_t;
  const float* sin_t;
  const float* gq;           // null: no per-head norm
  const float* gk;
  float eps;
  int window;                // > 0: keys j with slot - window < j <= slot only (sliding window)
  // rows of a mixed step (seq_idx set): the blocks of kFlashRows / G rows that
  // rows_uniform accepts are attn_prefill's; the row-wise kernel skips them
  int flash_rows;
};

// Query rows per attn_prefill CTA (query tokens x the G heads of a KV head).
constexpr int kFlashRows = 128;

// Rows t0 .. t0 + n - 1 of a mixed step are consecutive positions of one
// sequence, all inside the cache.  Every lane of the calling warp gets the same
// answer.
__device__ __forceinline__ bool rows_uniform(const int32_t* seq, const int32_t* pos, int t0, int n,
                                             const CacheView& c) {
  const int s0 = seq[t0], p0 = pos[t0];
  bool ok = s0 >= 0 && s0 < c.max_seq && p0 >= 0 && p0 + n <= c.max_ctx;
  for (int i = (int)(threadIdx.x & 31u); i < n; i += 32) ok = ok && seq[t0 + i] == s0 && pos[t0 + i] == p0 + i;
  return __all_sync(0xffffffffu, ok);
}

cudaError_t launch_rope_append(int kvtype, int hd, const RopeArgs& a, cudaStream_t s);
// prefill attention over an f16 cache (attn_prefill.cu): T query rows of one
// sequence (a.seq_fixed) at positions pos_base.., their K/V already appended;
// kmap/vmap from encode_kv_map over this layer's caches
cudaError_t encode_kv_map(CUtensorMap* map, const void* layer_base, int hd, const CacheView& c, int max_batch);
cudaError_t launch_attn_prefill(int hd, int G, const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a,
                                cudaStream_t s);
// f16 caches: kmap / vmap are the layer's tensor maps (encode_kv_map); f32: unused.
cudaError_t launch_attn_decode(int kvtype, int hd, int G, const CUtensorMap* kmap, const CUtensorMap* vmap,
                               const AttnArgs& a, cudaStream_t s);
// one-time per-kernel attributes (dynamic shared memory); call outside stream capture
cudaError_t attn_prepare(int kvtype, int hd, int G);

// set the calling thread's tq_last_error() message (api.cu)
void record_error(const char* msg);

// temperature / top-p sampling of logits [n][V] (sample.cu): per row a
// temperature (0: argmax), a top_p and a uniform number u in [0, 1)
cudaError_t launch_sample(const float* logits, int n, int V, const float* temperature, const float* top_p,
                          const float* u, int32_t* out, cudaStream_t s);

// out[b] = x[rows[b]] (rows of H floats), b < n
cudaError_t launch_gather_rows(const float* x, int H, int n_rows, const int32_t* rows, int n, float* out,
                               uint32_t* status, cudaStream_t s);

// argmax keys -> int32 indices
cudaError_t launch_argmax_finish(const unsigned long long* keys, int n, int32_t* out, cudaStream_t s);
// logits [n][V] -> per-row argmax, ties to the lowest index
// row argmax of [n][V] logits; softcap > 0 first replaces each logit by
// softcap * tanh(logit / softcap) in place
cudaError_t launch_argmax_rows(float* logits, int n, int V, float softcap, int32_t* out, cudaStream_t s);

}  // namespace tq
