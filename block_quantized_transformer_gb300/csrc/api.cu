// C ABI of libtq.so (declared in include/tq.h): argument checks on the host
// before anything is enqueued, the model object over caller-owned memory, the
// decode and prefill launch sequences, CUDA-graph replay of the decode step,
// and the status / poisoning rules of the tessl_torch README ("Handle
// ownership, closing and errors").
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "kernels.cuh"

namespace {

thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// formats of the tiled layout: Q4_0, AFFINE4, Q8_0
bool tiled_wtype(int32_t w) { return w == TQ_Q4_0 || w == TQ_AFFINE4 || w == TQ_Q8_0; }

constexpr int64_t kGemmPartFloats = 4 << 20;  // 16 MB of split-K partial sums
constexpr int kGemmCounters = 4096;

struct Layout {
  size_t x, qkv, att, act, act2, x16, inv_s, logits, xhead, cos_t, sin_t, part, counters, keys, status, chain_sync,
      gemm_part, gemm_ctr, bias, total;
  int T;                 // rows of activation buffers
  int split_dec, splits_dec, split_pf, splits_pf;
};

int qkv_width(const tq_config& c) { return (c.n_heads + 2 * c.n_kv_heads) * c.head_dim; }

bool validate(const tq_config* c) {
  if (c == nullptr) return set_error("config is NULL"), false;
  if (c->vocab <= 0 || c->hidden <= 0 || c->n_layers <= 0 || c->n_heads <= 0 ||
      c->n_kv_heads <= 0 || c->ffn <= 0)
    return set_error("config: sizes must be positive"), false;
  if (c->head_dim != 64 && c->head_dim != 128)
    return set_error("config: head_dim must be 64 or 128 (got %d)", c->head_dim), false;
  if (c->n_heads % c->n_kv_heads != 0)
    return set_error("config: n_heads must be a multiple of n_kv_heads"), false;
  const int G = c->n_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return set_error("config: n_heads / n_kv_heads must be 1, 2, 4 or 8 (got %d)", G), false;
  if (!tiled_wtype(c->wtype))
    return set_error("config: wtype must be TQ_Q4_0 (2), TQ_AFFINE4 (4) or TQ_Q8_0 (8)"), false;
  if (c->kvtype != TQ_KV_F32 && c->kvtype != TQ_KV_F16)
    return set_error("config: kvtype must be TQ_KV_F32 (0) or TQ_KV_F16 (1)"), false;
  const int ks[3] = {c->hidden, c->n_heads * c->head_dim, c->ffn};
  for (int k : ks)
    if (!tq::gemv_supported(k))
      return set_error("config: no GEMV thread mapping for an input width of %d "
                       "(need 32*kpt*p, kpt in 1..4, p in {8,...,128})", k), false;
  if (c->max_batch < 1 || c->max_ctx < 1 || c->max_prefill < 1)
    return set_error("config: max_batch, max_ctx and max_prefill must be >= 1"), false;
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f))
    return set_error("config: rms_eps and rope_theta must be positive"), false;
  if (c->arch < TQ_ARCH_QWEN3 || c->arch > TQ_ARCH_GEMMA3)
    return set_error("config: arch must be a tq_arch (0..3, got %d)", c->arch), false;
  if (c->sliding_window < 0 || c->sliding_pattern < 0 || !(c->logit_softcap >= 0.f) ||
      !(c->logit_softcap < 3.0e38f))
    return set_error("config: sliding_window, sliding_pattern and logit_softcap must be >= 0"), false;
  if (c->arch != TQ_ARCH_GEMMA3 && (c->sliding_window != 0 || c->sliding_pattern != 0 || c->logit_softcap != 0.f))
    return set_error("config: sliding_window, sliding_pattern and logit_softcap are gemma3's (set them to 0)"),
           false;
  if (c->page_size < 0) return set_error("config: page_size must be >= 0"), false;
  if (c->page_size > 0) {
    if (c->page_size % 32 != 0) return set_error("config: page_size must be a multiple of 32"), false;
    if (c->max_ctx % c->page_size != 0)
      return set_error("config: max_ctx must be a multiple of page_size"), false;
    if (c->n_pages < 1) return set_error("config: n_pages must be >= 1"), false;
  }
  return true;
}

Layout layout_of(const tq_config& c) {
  Layout L{};
  const int G = c.n_heads / c.n_kv_heads;
  L.T = c.max_batch > c.max_prefill ? c.max_batch : c.max_prefill;
  L.split_dec = 128 * (1 + (c.max_ctx - 1) / 8192);
  L.splits_dec = (c.max_ctx + L.split_dec - 1) / L.split_dec;
  L.split_pf = 1024;
  L.splits_pf = (c.max_ctx + L.split_pf - 1) / L.split_pf;
  const size_t part_dec = (size_t)c.max_batch * c.n_kv_heads * L.splits_dec;
  const size_t part_pf = (size_t)c.max_prefill * c.n_kv_heads * L.splits_pf;
  const size_t part_rows = part_dec > part_pf ? part_dec : part_pf;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.x = take((size_t)L.T * c.hidden * 4);
  L.qkv = take((size_t)L.T * qkv_width(c) * 4);
  L.att = take((size_t)L.T * c.n_heads * c.head_dim * 4);
  L.act = take((size_t)L.T * c.ffn * 4);
  // GEMM path (prefill, batched decode): rows of [gate | up], and the fp16
  // rows of the widest GEMM input with their scales
  const int kmax = std::max(c.hidden, std::max(c.n_heads * c.head_dim, c.ffn));
  L.act2 = take((size_t)L.T * 2 * c.ffn * 4);
  L.x16 = take((size_t)L.T * kmax * 2);
  L.inv_s = take((size_t)L.T * 4);
  L.logits = c.max_batch > 1 ? take((size_t)c.max_batch * c.vocab * 4) : 0;
  L.xhead = take((size_t)c.max_batch * c.hidden * 4);  // tq_step: each sequence's last row
  L.cos_t = take((size_t)c.max_ctx * (c.head_dim / 2) * 4);
  L.sin_t = take((size_t)c.max_ctx * (c.head_dim / 2) * 4);
  L.part = take(part_rows * G * (c.head_dim + 2) * 4);
  L.counters = take((size_t)L.T * c.n_kv_heads * 4);
  L.keys = take((size_t)L.T * 8);
  L.status = take(16);
  L.chain_sync = take((tq::kMaxPhases + 1) * 4);
  // split-K partial sums of the GEMMs over few rows (batched decode)
  L.gemm_part = L.T > 1 ? take((size_t)kGemmPartFloats * 4) : 0;
  L.gemm_ctr = L.T > 1 ? take((size_t)kGemmCounters * 4) : 0;
  // qwen2: each layer's q, k and v biases side by side, as the Q/K/V output rows
  L.bias = c.arch == TQ_ARCH_QWEN2 ? take((size_t)c.n_layers * qkv_width(c) * 4) : 0;
  L.total = off;
  return L;
}

size_t kv_bytes(const tq_config& c) {
  const size_t esz = c.kvtype == TQ_KV_F16 ? 2 : 4;
  const size_t per_layer =
      c.page_size > 0 ? (size_t)c.n_pages * c.n_kv_heads * c.page_size * c.head_dim
                      : (size_t)c.max_batch * c.n_kv_heads * c.max_ctx * c.head_dim;
  return (size_t)c.n_layers * per_layer * esz;
}

bool check_qmat(const tq_qmat& m, const char* name) {
  if (m.qs_dev == nullptr || m.d_dev == nullptr) return set_error("weights: %s is NULL", name), false;
  if (!aligned16(m.qs_dev) || !aligned16(m.d_dev))
    return set_error("weights: %s must be 16-byte aligned", name), false;
  return true;
}

}  // namespace

namespace tq {
void record_error(const char* msg) { set_error("%s", msg); }
}  // namespace tq

struct tq_model {
  tq_config cfg;
  std::vector<tq_layer> layers;
  tq_qmat embd, head;
  const float* out_norm;
  uint8_t* ws;
  Layout L;
  void* kc;
  void* vc;
  size_t layer_kv_bytes;
  bool poisoned = false;
  std::string poison_reason;
  unsigned chain_wait_limit = 0;  // polls of a chain's grid-wide waits (0: the kernel's default)
  std::vector<CUtensorMap> kmap, vmap;  // per layer, f16 caches: tensor maps of the prefill attention
  // decode-step graph
  cudaGraphExec_t gexec = nullptr;
  struct {
    int batch;
    const void* p[6];
    void* stream;
  } gkey{};

  float* x() const { return reinterpret_cast<float*>(ws + L.x); }
  float* qkv() const { return reinterpret_cast<float*>(ws + L.qkv); }
  float* att() const { return reinterpret_cast<float*>(ws + L.att); }
  float* act() const { return reinterpret_cast<float*>(ws + L.act); }
  float* act2() const { return reinterpret_cast<float*>(ws + L.act2); }
  __half* x16() const { return reinterpret_cast<__half*>(ws + L.x16); }
  float* inv_s() const { return reinterpret_cast<float*>(ws + L.inv_s); }
  float* logits_ws() const { return reinterpret_cast<float*>(ws + L.logits); }
  float* xhead() const { return reinterpret_cast<float*>(ws + L.xhead); }
  float* cos_t() const { return reinterpret_cast<float*>(ws + L.cos_t); }
  float* sin_t() const { return reinterpret_cast<float*>(ws + L.sin_t); }
  float* part() const { return reinterpret_cast<float*>(ws + L.part); }
  unsigned* counters() const { return reinterpret_cast<unsigned*>(ws + L.counters); }
  unsigned long long* keys() const { return reinterpret_cast<unsigned long long*>(ws + L.keys); }
  uint32_t* status() const { return reinterpret_cast<uint32_t*>(ws + L.status); }
  unsigned* chain_sync() const { return reinterpret_cast<unsigned*>(ws + L.chain_sync); }
  float* gemm_part() const { return L.T > 1 ? reinterpret_cast<float*>(ws + L.gemm_part) : nullptr; }
  unsigned* gemm_ctr() const { return L.T > 1 ? reinterpret_cast<unsigned*>(ws + L.gemm_ctr) : nullptr; }
  void* kc_layer(int l) const { return static_cast<uint8_t*>(kc) + (size_t)l * layer_kv_bytes; }
  const float* qkv_bias(int l) const {
    return cfg.arch == TQ_ARCH_QWEN2 ? reinterpret_cast<const float*>(ws + L.bias) + (size_t)l * qkv_width(cfg)
                                     : nullptr;
  }
  bool qk_norm() const { return cfg.arch == TQ_ARCH_QWEN3 || cfg.arch == TQ_ARCH_GEMMA3; }
  int gate_act() const { return cfg.arch == TQ_ARCH_GEMMA3 ? tq::ACT_GELU_TANH : tq::ACT_SILU; }
  // sliding window of layer l (0: the whole context)
  int window(int l) const {
    if (cfg.arch != TQ_ARCH_GEMMA3 || cfg.sliding_window <= 0) return 0;
    const int p = cfg.sliding_pattern;
    return p > 0 && l % p == p - 1 ? 0 : cfg.sliding_window;
  }
  void* vc_layer(int l) const { return static_cast<uint8_t*>(vc) + (size_t)l * layer_kv_bytes; }
};

namespace {

tq_status fail_cuda(tq_model* m, cudaError_t e, const char* what) {
  set_error("%s: CUDA error %s (%s); the model is poisoned: free it and create a new one",
            what, cudaGetErrorName(e), cudaGetErrorString(e));
  (void)cudaGetLastError();  // the error is reported here; do not leave it for the caller's next call
  if (m != nullptr) {
    m->poisoned = true;
    m->poison_reason = g_last_error;
  }
  return TQ_INTERNAL;
}

bool refuse_if_poisoned(tq_model* m) {
  if (m == nullptr) return set_error("model is NULL"), true;
  if (m->poisoned) {
    set_error("model is poisoned (%s); recreate it", m->poison_reason.c_str());
    return true;
  }
  return false;
}

tq::GemvSeg seg_of(const tq_qmat& q, int rows) {
  return tq::GemvSeg{static_cast<const uint8_t*>(q.qs_dev), q.d_dev, rows};
}

tq::CacheView cache_view(const tq_model* m, const int32_t* block_table) {
  const tq_config& c = m->cfg;
  tq::CacheView v{};
  v.max_ctx = c.max_ctx;
  v.max_seq = c.max_batch;
  v.n_kv = c.n_kv_heads;
  v.page_size = c.page_size;
  v.n_pages = c.n_pages;
  v.block_table = block_table;
  v.bt_stride = c.page_size > 0 ? c.max_ctx / c.page_size : 0;
  return v;
}

// Layer l's tensor map of the K (V) cache; null for an f32 cache.
const CUtensorMap* kv_map(const tq_model* m, int l, bool v) {
  if (m->kmap.empty()) return nullptr;
  return v ? &m->vmap[l] : &m->kmap[l];
}

// The layer loop shared by decode (T = batch, one token per sequence) and
// prefill (T tokens of sequence `seq` at positions pos_base..).
// GEMV arguments of the projections of layer l over T token rows.
tq::GemvArgs qkv_args(const tq_model* m, int l, int T) {
  const tq_config& c = m->cfg;
  const tq_layer& ly = m->layers[l];
  tq::GemvArgs g{};  // RMSNorm + Q/K/V projections
  g.seg[0] = seg_of(ly.attn_q, c.n_heads * c.head_dim);
  g.seg[1] = seg_of(ly.attn_k, c.n_kv_heads * c.head_dim);
  g.seg[2] = seg_of(ly.attn_v, c.n_kv_heads * c.head_dim);
  g.nseg = 3;
  g.K = c.hidden;
  g.N = qkv_width(c);
  g.B = T;
  g.x = m->x();
  g.gain = ly.attn_norm_dev;
  g.eps = c.rms_eps;
  g.y = m->qkv();
  g.status = m->status();
  g.bias = m->qkv_bias(l);
  return g;
}

tq::GemvArgs out_args(const tq_model* m, int l, int T) {
  const tq_config& c = m->cfg;
  tq::GemvArgs o{};  // output projection + residual
  o.seg[0] = seg_of(m->layers[l].attn_output, c.hidden);
  o.nseg = 1;
  o.K = c.n_heads * c.head_dim;
  o.N = c.hidden;
  o.B = T;
  o.x = m->att();
  o.y = m->x();
  o.residual = m->x();
  o.status = m->status();
  return o;
}

tq::GemvArgs ffn_args(const tq_model* m, int l, int T) {
  const tq_config& c = m->cfg;
  const tq_layer& ly = m->layers[l];
  tq::GemvArgs f{};  // RMSNorm + gate/up + SwiGLU
  f.seg[0] = seg_of(ly.ffn_gate, c.ffn);
  f.seg[1] = seg_of(ly.ffn_up, c.ffn);
  f.nseg = 2;
  f.K = c.hidden;
  f.N = c.ffn;
  f.B = T;
  f.x = m->x();
  f.gain = ly.ffn_norm_dev;
  f.eps = c.rms_eps;
  f.y = m->act();
  f.status = m->status();
  f.act = m->gate_act();
  return f;
}

tq::GemvArgs down_args(const tq_model* m, int l, int T) {
  const tq_config& c = m->cfg;
  tq::GemvArgs d{};  // down projection + residual
  d.seg[0] = seg_of(m->layers[l].ffn_down, c.hidden);
  d.nseg = 1;
  d.K = c.ffn;
  d.N = c.hidden;
  d.B = T;
  d.x = m->act();
  d.y = m->x();
  d.residual = m->x();
  d.status = m->status();
  return d;
}

tq::GemvArgs head_args(const tq_model* m, const float* x, int B, float* logits) {
  const tq_config& c = m->cfg;
  tq::GemvArgs h{};  // final RMSNorm + tied LM head + argmax
  h.seg[0] = seg_of(m->head, c.vocab);
  h.nseg = 1;
  h.K = c.hidden;
  h.N = c.vocab;
  h.B = B;
  h.x = x;
  h.gain = m->out_norm;
  h.eps = c.rms_eps;
  h.y = logits;
  h.argmax_keys = m->keys();
  h.status = m->status();
  h.softcap = c.logit_softcap;
  return h;
}

tq::RopeArgs rope_args(const tq_model* m, int l, int T, const int32_t* pos, const int32_t* kv_len, int pos_base,
                       int seq_fixed, const int32_t* block_table, const int32_t* seq_idx = nullptr) {
  const tq_config& c = m->cfg;
  tq::RopeArgs r{};
  r.qkv = m->qkv();
  r.T = T;
  r.nq = c.n_heads;
  r.nkv = c.n_kv_heads;
  r.pos = pos;
  r.kv_len = kv_len;
  r.pos_base = pos_base;
  r.seq_fixed = seq_fixed;
  r.seq_idx = seq_idx;
  r.kc = m->kc_layer(l);
  r.vc = m->vc_layer(l);
  r.cache = cache_view(m, block_table);
  r.cos_t = m->cos_t();
  r.sin_t = m->sin_t();
  r.gq = m->qk_norm() ? m->layers[l].attn_q_norm_dev : nullptr;
  r.gk = m->qk_norm() ? m->layers[l].attn_k_norm_dev : nullptr;
  r.eps = c.rms_eps;
  r.status = m->status();
  return r;
}

tq::AttnArgs attn_args(const tq_model* m, int l, int T, const int32_t* pos, const int32_t* kv_len, int pos_base,
                       int seq_fixed, const int32_t* block_table, bool prefill, const int32_t* seq_idx = nullptr) {
  const tq_config& c = m->cfg;
  const int hd = c.head_dim;
  tq::AttnArgs a{};
  a.q = m->qkv();
  a.q_stride = qkv_width(c);
  a.o = m->att();
  a.T = T;
  a.nq = c.n_heads;
  a.nkv = c.n_kv_heads;
  a.kv_len = kv_len;
  a.pos_base = pos_base;
  a.seq_fixed = seq_fixed;
  a.seq_idx = seq_idx;
  a.kc = m->kc_layer(l);
  a.vc = m->vc_layer(l);
  a.cache = cache_view(m, block_table);
  a.split_keys = prefill ? m->L.split_pf : m->L.split_dec;
  a.max_splits = prefill ? m->L.splits_pf : m->L.splits_dec;
  a.part = m->part();
  a.counters = m->counters();
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)hd));
  a.status = m->status();
  a.fused = prefill ? 0 : 1;
  a.pos = pos;
  a.cos_t = m->cos_t();
  a.sin_t = m->sin_t();
  a.gq = m->qk_norm() ? m->layers[l].attn_q_norm_dev : nullptr;
  a.gk = m->qk_norm() ? m->layers[l].attn_k_norm_dev : nullptr;
  a.eps = c.rms_eps;
  a.window = m->window(l);
  return a;
}

cudaError_t gemm_prep(tq_model* m, int T, const float* x, const float* up, int K, const float* gain, cudaStream_t s,
                      int ldx = 0) {
  tq::XPrep16Args p{};
  p.x = x;
  p.up = up;
  p.act = m->gate_act();
  p.ldx = ldx > 0 ? ldx : K;
  p.gain = gain;
  p.eps = m->cfg.rms_eps;
  p.K = K;
  p.T = T;
  p.x16 = m->x16();
  p.inv_s = m->inv_s();
  return tq::launch_xprep16(p, s);
}

cudaError_t gemm_run(tq_model* m, int T, const tq::GemvSeg* seg, int nseg, int K, float* y, int ldy,
                     const float* residual, cudaStream_t s, const float* bias = nullptr) {
  tq::TcGemmArgs g{};
  for (int i = 0; i < nseg; ++i) g.seg[i] = seg[i];
  g.nseg = nseg;
  g.K = K;
  g.T = T;
  g.x16 = m->x16();
  g.inv_s = m->inv_s();
  g.y = y;
  g.ldy = ldy;
  g.residual = residual;
  g.bias = bias;
  g.status = m->status();
  g.part = m->gemm_part();
  g.part_cap = kGemmPartFloats;
  g.counters = m->gemm_ctr();
  g.n_counters = kGemmCounters;
  return tq::launch_tcgemm(m->cfg.wtype, g, s);
}

// The layers for T >= 2 token rows with every projection as a tensor-core
// GEMM over all rows (each weight tile decoded once per CTA of up to 256
// rows), each phase's input turned into fp16 rows by one xprep16 launch.
//  - prefill (pos == nullptr): rows of one sequence at pos_base..; the K/V of
//    all rows are appended first, then each row attends over its causal prefix;
//  - mixed (seq_idx != nullptr): row t is a token of sequence seq_idx[t] at
//    position pos[t] (its cache slot too), rows of a sequence in position
//    order; appended first as well, then each row attends over its own prefix;
//  - batched decode: row b is sequence b at positions[b]; QK-norm, RoPE and
//    the append happen inside the fused attention.
cudaError_t run_layers_gemm(tq_model* m, int T, const int32_t* pos, const int32_t* kv_len, int pos_base,
                            int seq_fixed, const int32_t* block_table, cudaStream_t s,
                            const int32_t* seq_idx = nullptr) {
  const tq_config& c = m->cfg;
  const int hd = c.head_dim, nq = c.n_heads, nkv = c.n_kv_heads, G = nq / nkv;
  const bool mixed = seq_idx != nullptr;
  const bool prefill = pos == nullptr || mixed;
  cudaError_t e;
  for (int l = 0; l < c.n_layers; ++l) {
    const tq_layer& ly = m->layers[l];
    const tq::GemvSeg qkv[3] = {seg_of(ly.attn_q, nq * hd), seg_of(ly.attn_k, nkv * hd), seg_of(ly.attn_v, nkv * hd)};
    if ((e = gemm_prep(m, T, m->x(), nullptr, c.hidden, ly.attn_norm_dev, s)) != cudaSuccess) return e;
    e = gemm_run(m, T, qkv, 3, c.hidden, m->qkv(), qkv_width(c), nullptr, s, m->qkv_bias(l));
    if (e != cudaSuccess) return e;
    if (prefill) {
      const tq::RopeArgs r = rope_args(m, l, T, pos, kv_len, pos_base, seq_fixed, block_table, seq_idx);
      if ((e = tq::launch_rope_append(c.kvtype, hd, r, s)) != cudaSuccess) return e;
    }
    const tq::AttnArgs a = attn_args(m, l, T, pos, kv_len, pos_base, seq_fixed, block_table, prefill, seq_idx);
    if (prefill && !mixed && c.kvtype == TQ_KV_F16) {
      // prefill over an f16 cache: flash-attention tiles staged by tensor maps
      // of this layer's caches (made at model creation; a paged cache's block
      // table is read in the kernel)
      e = tq::launch_attn_prefill(hd, G, m->kmap[l], m->vmap[l], a, s);
    } else if (mixed && c.kvtype == TQ_KV_F16) {
      // mixed rows over an f16 cache: blocks of rows that are one sequence's
      // consecutive positions (prompt chunks) take the flash kernel, the
      // other rows (decode tokens, a chunk's ragged ends) the row-wise kernel
      tq::AttnArgs af = a;
      af.flash_rows = 1;
      e = tq::launch_attn_prefill(hd, G, m->kmap[l], m->vmap[l], af, s);
      if (e == cudaSuccess) e = tq::launch_attn_decode(c.kvtype, hd, G, kv_map(m, l, false), kv_map(m, l, true), af, s);
    } else {
      e = tq::launch_attn_decode(c.kvtype, hd, G, kv_map(m, l, false), kv_map(m, l, true), a, s);
    }
    if (e != cudaSuccess) return e;
    const tq::GemvSeg o = seg_of(ly.attn_output, c.hidden);
    if ((e = gemm_prep(m, T, m->att(), nullptr, nq * hd, nullptr, s)) != cudaSuccess) return e;
    if ((e = gemm_run(m, T, &o, 1, nq * hd, m->x(), c.hidden, m->x(), s)) != cudaSuccess) return e;
    const tq::GemvSeg gate = seg_of(ly.ffn_gate, c.ffn), up = seg_of(ly.ffn_up, c.ffn);
    if ((e = gemm_prep(m, T, m->x(), nullptr, c.hidden, ly.ffn_norm_dev, s)) != cudaSuccess) return e;
    // gate and up in one GEMM: row t of act2 holds [gate | up]
    const tq::GemvSeg gu[2] = {gate, up};
    if ((e = gemm_run(m, T, gu, 2, c.hidden, m->act2(), 2 * c.ffn, nullptr, s)) != cudaSuccess) return e;
    const tq::GemvSeg down = seg_of(ly.ffn_down, c.hidden);
    if ((e = gemm_prep(m, T, m->act2(), m->act2() + c.ffn, c.ffn, nullptr, s, 2 * c.ffn)) != cudaSuccess) return e;
    if ((e = gemm_run(m, T, &down, 1, c.ffn, m->x(), c.hidden, m->x(), s)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Greedy head on one row: the one-phase GEMV chain with the argmax epilogue.
cudaError_t run_head_one(tq_model* m, const float* x, float* logits, int32_t* argmax, cudaStream_t s) {
  tq::GemvChain ch{};
  ch.ph[0] = head_args(m, x, 1, logits);
  ch.mode[0] = tq::GEMV_ARGMAX;
  ch.n = 1;
  cudaError_t e = tq::launch_gemv_chain(m->cfg.wtype, ch, s);
  if (e != cudaSuccess) return e;
  return tq::launch_argmax_finish(m->keys(), 1, argmax, s);
}

// Greedy head on B >= 2 rows of x: final RMSNorm + LM head as a GEMM into
// the logits (the caller's, or the workspace's), then a row argmax.
cudaError_t run_head_gemm(tq_model* m, const float* x, int B, float* logits, int32_t* argmax, cudaStream_t s) {
  const tq_config& c = m->cfg;
  float* lg = logits != nullptr ? logits : m->logits_ws();
  const tq::GemvSeg h = seg_of(m->head, c.vocab);
  cudaError_t e = gemm_prep(m, B, x, nullptr, c.hidden, m->out_norm, s);
  if (e == cudaSuccess) e = gemm_run(m, B, &h, 1, c.hidden, lg, c.vocab, nullptr, s);
  if (e == cudaSuccess) e = tq::launch_argmax_rows(lg, B, c.vocab, c.logit_softcap, argmax, s);
  return e;
}

// The GEMV chain that follows layer l's attention: output projection +
// residual, RMSNorm + gate/up + SwiGLU, down projection + residual, then the
// next layer's RMSNorm + Q/K/V (after the last layer: final norm + LM head +
// argmax keys over `head_B` rows at head_x).
tq::GemvChain layer_chain(const tq_model* m, int l, int T, const float* head_x, int head_B, float* logits) {
  const tq_config& c = m->cfg;
  tq::GemvChain ch{};
  ch.ph[0] = out_args(m, l, T);
  ch.mode[0] = tq::GEMV_STORE;
  ch.ph[1] = ffn_args(m, l, T);
  ch.mode[1] = tq::GEMV_SWIGLU;
  ch.ph[2] = down_args(m, l, T);
  ch.mode[2] = tq::GEMV_STORE;
  if (l + 1 < c.n_layers) {
    ch.ph[3] = qkv_args(m, l + 1, T);
    ch.mode[3] = tq::GEMV_STORE;
  } else {
    ch.ph[3] = head_args(m, head_x, head_B, logits);
    ch.mode[3] = tq::GEMV_ARGMAX;
  }
  ch.n = 4;
  ch.sync = m->chain_sync();
  ch.sync_limit = m->chain_wait_limit;
  return ch;
}

// The layers and the head.  The GEMVs between two attention launches run as
// one persistent chain: output projection, gate/up, down projection of layer
// l and the Q/K/V projection of layer l+1 (the LM head after the last layer),
// so the weight stream does not drain between them.  `head_x`/`head_B`: the
// rows the head reads (all decode rows; the last prompt token in prefill).
cudaError_t run_layers(tq_model* m, int T, const int32_t* pos, const int32_t* kv_len, int pos_base,
                       int seq_fixed, const int32_t* block_table, bool prefill, const float* head_x,
                       int head_B, float* logits, int32_t* argmax, cudaStream_t s) {
  const tq_config& c = m->cfg;
  const int hd = c.head_dim, nq = c.n_heads, nkv = c.n_kv_heads, G = nq / nkv;
  cudaError_t e;
  {
    tq::GemvChain ch{};
    ch.ph[0] = qkv_args(m, 0, T);
    ch.mode[0] = tq::GEMV_STORE;
    ch.n = 1;
    if ((e = tq::launch_gemv_chain(c.wtype, ch, s)) != cudaSuccess) return e;
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const tq_layer& ly = m->layers[l];
    // QK-norm + RoPE + KV append: its own kernel in prefill (every token's K/V
    // must be stored before any token attends); inside attention in decode
    if (prefill) {
      const tq::RopeArgs r = rope_args(m, l, T, pos, kv_len, pos_base, seq_fixed, block_table);
      if ((e = tq::launch_rope_append(c.kvtype, hd, r, s)) != cudaSuccess) return e;
    }
    const tq::AttnArgs a = attn_args(m, l, T, pos, kv_len, pos_base, seq_fixed, block_table, prefill);
    e = tq::launch_attn_decode(c.kvtype, hd, G, kv_map(m, l, false), kv_map(m, l, true), a, s);
    if (e != cudaSuccess) return e;
    // output projection, FFN, and the next layer's Q/K/V (or the head)
    const tq::GemvChain ch = layer_chain(m, l, T, head_x, head_B, logits);
    if ((e = tq::launch_gemv_chain(c.wtype, ch, s)) != cudaSuccess) return e;
  }
  return tq::launch_argmax_finish(m->keys(), head_B, argmax, s);
}

cudaError_t enqueue_decode(tq_model* m, int batch, const int32_t* tokens, const int32_t* positions,
                           const int32_t* kv_lens, const int32_t* block_table, float* logits,
                           int32_t* argmax, cudaStream_t s) {
  const tq_config& c = m->cfg;
  cudaError_t e = tq::launch_embed(c.wtype, m->embd.qs_dev, m->embd.d_dev, c.vocab, c.hidden, tokens,
                                   batch, m->x(), m->status(), m->keys(), batch, s);
  if (e != cudaSuccess) return e;
  if (batch >= 2) {  // batched: weights read once per 32 sequences
    e = run_layers_gemm(m, batch, positions, kv_lens, 0, -1, block_table, s);
    return e == cudaSuccess ? run_head_gemm(m, m->x(), batch, logits, argmax, s) : e;
  }
  return run_layers(m, batch, positions, kv_lens, 0, -1, block_table, false, m->x(), batch, logits,
                    argmax, s);
}

}  // namespace

extern "C" {

const char* tq_last_error(void) { return g_last_error.c_str(); }

size_t tq_workspace_bytes(const tq_config* cfg) {
  if (!validate(cfg)) return 0;
  return layout_of(*cfg).total;
}

size_t tq_kv_cache_bytes(const tq_config* cfg) {
  if (!validate(cfg)) return 0;
  return kv_bytes(*cfg);
}

tq_status tq_model_create(const tq_config* cfg, const tq_weights* w, void* workspace, void* k_cache,
                          void* v_cache, tq_model** out) {
  if (out == nullptr) return set_error("out is NULL"), TQ_REFUSED;
  *out = nullptr;
  if (!validate(cfg)) return TQ_REFUSED;
  if (w == nullptr || w->layers == nullptr) return set_error("weights or weights->layers is NULL"), TQ_REFUSED;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return set_error("workspace must be non-NULL and 256-byte aligned"), TQ_REFUSED;
  if (k_cache == nullptr || v_cache == nullptr || !aligned16(k_cache) || !aligned16(v_cache))
    return set_error("k_cache and v_cache must be non-NULL and 16-byte aligned"), TQ_REFUSED;
  if (!check_qmat(w->token_embd, "token_embd")) return TQ_REFUSED;
  if (w->output.qs_dev != nullptr && !check_qmat(w->output, "output")) return TQ_REFUSED;
  if (w->output_norm_dev == nullptr) return set_error("weights: output_norm is NULL"), TQ_REFUSED;
  for (int l = 0; l < cfg->n_layers; ++l) {
    const tq_layer& ly = w->layers[l];
    const tq_qmat* mats[7] = {&ly.attn_q, &ly.attn_k, &ly.attn_v, &ly.attn_output,
                              &ly.ffn_gate, &ly.ffn_up, &ly.ffn_down};
    for (int i = 0; i < 7; ++i) {
      char name[64];
      snprintf(name, sizeof(name), "blk.%d matrix %d", l, i);
      if (!check_qmat(*mats[i], name)) return TQ_REFUSED;
    }
    const bool qk_norm = cfg->arch == TQ_ARCH_QWEN3 || cfg->arch == TQ_ARCH_GEMMA3;
    if (!ly.attn_norm_dev || !ly.ffn_norm_dev || (qk_norm && (!ly.attn_q_norm_dev || !ly.attn_k_norm_dev)))
      return set_error("weights: a gain of blk.%d is NULL", l), TQ_REFUSED;
    const float* gs[4] = {ly.attn_norm_dev, ly.ffn_norm_dev, qk_norm ? ly.attn_q_norm_dev : nullptr,
                          qk_norm ? ly.attn_k_norm_dev : nullptr};
    for (const float* gp : gs)
      if (!aligned16(gp)) return set_error("weights: gains of blk.%d must be 16-byte aligned", l), TQ_REFUSED;
    if (cfg->arch == TQ_ARCH_QWEN2 && (!ly.attn_q_bias_dev || !ly.attn_k_bias_dev || !ly.attn_v_bias_dev))
      return set_error("weights: qwen2 needs the q, k and v biases of blk.%d", l), TQ_REFUSED;
  }
  if (!aligned16(w->output_norm_dev)) return set_error("weights: output_norm must be 16-byte aligned"), TQ_REFUSED;

  tq_model* m = new tq_model();
  m->cfg = *cfg;
  m->layers.assign(w->layers, w->layers + cfg->n_layers);
  m->embd = w->token_embd;
  m->head = w->output.qs_dev != nullptr ? w->output : w->token_embd;
  m->out_norm = w->output_norm_dev;
  m->ws = static_cast<uint8_t*>(workspace);
  m->L = layout_of(*cfg);
  m->kc = k_cache;
  m->vc = v_cache;
  m->layer_kv_bytes = kv_bytes(*cfg) / cfg->n_layers;

  // RoPE table in double precision on the host: angle = pos * theta^(-i/half)
  const int half = cfg->head_dim / 2;
  std::vector<float> cs((size_t)cfg->max_ctx * half), sn((size_t)cfg->max_ctx * half);
  for (int p = 0; p < cfg->max_ctx; ++p)
    for (int i = 0; i < half; ++i) {
      const double inv = 1.0 / std::pow((double)cfg->rope_theta, (double)i / (double)half);
      const double ang = (double)p * inv;
      cs[(size_t)p * half + i] = (float)std::cos(ang);
      sn[(size_t)p * half + i] = (float)std::sin(ang);
    }
  cudaError_t e = tq::attn_prepare(cfg->kvtype, cfg->head_dim, cfg->n_heads / cfg->n_kv_heads);
  if (e == cudaSuccess && cfg->kvtype == TQ_KV_F16) {
    m->kmap.resize(cfg->n_layers);
    m->vmap.resize(cfg->n_layers);
    const tq::CacheView cv = cache_view(m, nullptr);
    for (int l = 0; l < cfg->n_layers && e == cudaSuccess; ++l) {
      e = tq::encode_kv_map(&m->kmap[l], m->kc_layer(l), cfg->head_dim, cv, cfg->max_batch);
      if (e == cudaSuccess) e = tq::encode_kv_map(&m->vmap[l], m->vc_layer(l), cfg->head_dim, cv, cfg->max_batch);
    }
  }
  if (e == cudaSuccess) e = cudaMemset(workspace, 0, m->L.total);
  if (cfg->arch == TQ_ARCH_QWEN2)  // [bq | bk | bv] of each layer, in the order of the Q/K/V rows
    for (int l = 0; l < cfg->n_layers && e == cudaSuccess; ++l) {
      float* b = const_cast<float*>(m->qkv_bias(l));
      const size_t nq = (size_t)cfg->n_heads * cfg->head_dim, nk = (size_t)cfg->n_kv_heads * cfg->head_dim;
      e = cudaMemcpy(b, w->layers[l].attn_q_bias_dev, nq * 4, cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess) e = cudaMemcpy(b + nq, w->layers[l].attn_k_bias_dev, nk * 4, cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess)
        e = cudaMemcpy(b + nq + nk, w->layers[l].attn_v_bias_dev, nk * 4, cudaMemcpyDeviceToDevice);
    }
  if (e == cudaSuccess) e = cudaMemcpy(m->cos_t(), cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(m->sin_t(), sn.data(), sn.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    fail_cuda(nullptr, e, "tq_model_create");
    delete m;
    return TQ_INTERNAL;
  }
  *out = m;
  return TQ_OK;
}

tq_status tq_prefill(tq_model* m, int32_t seq, const int32_t* tokens, int32_t n_tokens,
                     int32_t start_pos, const int32_t* block_table, float* logits, int32_t* argmax,
                     void* stream) {
  if (refuse_if_poisoned(m)) return TQ_REFUSED;
  const tq_config& c = m->cfg;
  if (tokens == nullptr || argmax == nullptr) return set_error("tokens and argmax must not be NULL"), TQ_REFUSED;
  if (n_tokens < 1 || n_tokens > c.max_prefill)
    return set_error("n_tokens=%d outside [1, max_prefill=%d]", n_tokens, c.max_prefill), TQ_REFUSED;
  if (start_pos < 0 || (int64_t)start_pos + n_tokens > c.max_ctx)
    return set_error("start_pos=%d + n_tokens=%d exceeds max_ctx=%d", start_pos, n_tokens, c.max_ctx),
           TQ_REFUSED;
  if (c.page_size > 0) {
    if (block_table == nullptr) return set_error("paged cache: block_table must not be NULL"), TQ_REFUSED;
    seq = 0;
  } else if (seq < 0 || seq >= c.max_batch) {
    return set_error("seq=%d outside [0, max_batch=%d)", seq, c.max_batch), TQ_REFUSED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = tq::launch_embed(c.wtype, m->embd.qs_dev, m->embd.d_dev, c.vocab, c.hidden, tokens,
                                   n_tokens, m->x(), m->status(), m->keys(), 1, s);
  if (e == cudaSuccess && n_tokens >= 2) {
    e = run_layers_gemm(m, n_tokens, nullptr, nullptr, start_pos, seq, block_table, s);
    if (e == cudaSuccess) e = run_head_one(m, m->x() + (size_t)(n_tokens - 1) * c.hidden, logits, argmax, s);
  } else if (e == cudaSuccess) {
    e = run_layers(m, n_tokens, nullptr, nullptr, start_pos, seq, block_table, true,
                   m->x() + (size_t)(n_tokens - 1) * c.hidden, 1, logits, argmax, s);
  }
  if (e != cudaSuccess) return fail_cuda(m, e, "tq_prefill");
  return TQ_OK;
}

static tq_status check_decode_args(tq_model* m, int32_t batch, const int32_t* tokens,
                                   const int32_t* positions, const int32_t* kv_lens,
                                   const int32_t* block_table, int32_t* argmax) {
  if (refuse_if_poisoned(m)) return TQ_REFUSED;
  const tq_config& c = m->cfg;
  if (batch < 1 || batch > c.max_batch)
    return set_error("batch=%d outside [1, max_batch=%d]", batch, c.max_batch), TQ_REFUSED;
  if (!tokens || !positions || !kv_lens || !argmax)
    return set_error("tokens, positions, kv_lens and argmax must not be NULL"), TQ_REFUSED;
  if (c.page_size > 0 && block_table == nullptr)
    return set_error("paged cache: block_table must not be NULL"), TQ_REFUSED;
  return TQ_OK;
}

tq_status tq_decode_step(tq_model* m, int32_t batch, const int32_t* tokens, const int32_t* positions,
                         const int32_t* kv_lens, const int32_t* block_table, float* logits,
                         int32_t* argmax, void* stream) {
  tq_status st = check_decode_args(m, batch, tokens, positions, kv_lens, block_table, argmax);
  if (st != TQ_OK) return st;
  cudaError_t e = enqueue_decode(m, batch, tokens, positions, kv_lens,
                                 m->cfg.page_size > 0 ? block_table : nullptr, logits, argmax,
                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(m, e, "tq_decode_step");
  return TQ_OK;
}

tq_status tq_step(tq_model* m, int32_t n_rows, const int32_t* tokens, const int32_t* row_seq,
                  const int32_t* row_pos, int32_t n_seq, const int32_t* last_row, const int32_t* block_table,
                  float* logits, int32_t* argmax, void* stream) {
  if (refuse_if_poisoned(m)) return TQ_REFUSED;
  const tq_config& c = m->cfg;
  if (n_rows < 1 || n_rows > c.max_prefill)
    return set_error("n_rows=%d outside [1, max_prefill=%d]", n_rows, c.max_prefill), TQ_REFUSED;
  if (n_seq < 1 || n_seq > c.max_batch || n_seq > n_rows)
    return set_error("n_seq=%d outside [1, min(max_batch=%d, n_rows)]", n_seq, c.max_batch), TQ_REFUSED;
  if (!tokens || !row_seq || !row_pos || !last_row || !argmax)
    return set_error("tokens, row_seq, row_pos, last_row and argmax must not be NULL"), TQ_REFUSED;
  if (c.page_size > 0 && block_table == nullptr)
    return set_error("paged cache: block_table must not be NULL"), TQ_REFUSED;
  if (n_seq > 1 && logits == nullptr && m->L.logits == 0)
    return set_error("n_seq > 1 needs logits or a model with max_batch > 1"), TQ_REFUSED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t* bt = c.page_size > 0 ? block_table : nullptr;
  cudaError_t e = tq::launch_embed(c.wtype, m->embd.qs_dev, m->embd.d_dev, c.vocab, c.hidden, tokens, n_rows, m->x(),
                                   m->status(), m->keys(), n_seq, s);
  if (e == cudaSuccess) e = run_layers_gemm(m, n_rows, row_pos, row_pos, 0, -1, bt, s, row_seq);
  // the head reads each sequence's last row, gathered
  float* xl = m->xhead();
  if (e == cudaSuccess) e = tq::launch_gather_rows(m->x(), c.hidden, n_rows, last_row, n_seq, xl, m->status(), s);
  if (e == cudaSuccess)
    e = n_seq == 1 ? run_head_one(m, xl, logits, argmax, s) : run_head_gemm(m, xl, n_seq, logits, argmax, s);
  if (e != cudaSuccess) return fail_cuda(m, e, "tq_step");
  return TQ_OK;
}

tq_status tq_decode_step_graph(tq_model* m, int32_t batch, const int32_t* tokens,
                               const int32_t* positions, const int32_t* kv_lens,
                               const int32_t* block_table, float* logits, int32_t* argmax,
                               void* stream) {
  tq_status st = check_decode_args(m, batch, tokens, positions, kv_lens, block_table, argmax);
  if (st != TQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[6] = {tokens, positions, kv_lens, block_table, logits, argmax};
  bool same = m->gexec != nullptr && m->gkey.batch == batch && m->gkey.stream == stream;
  for (int i = 0; same && i < 6; ++i) same = m->gkey.p[i] == ptrs[i];
  cudaError_t e;
  if (!same) {
    if (m->gexec != nullptr) {
      cudaGraphExecDestroy(m->gexec);
      m->gexec = nullptr;
    }
    if (s == nullptr) return set_error("graph replay needs a non-default stream"), TQ_REFUSED;
    cudaGraph_t graph = nullptr;
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return fail_cuda(m, e, "tq_decode_step_graph: begin capture");
    cudaError_t le = enqueue_decode(m, batch, tokens, positions, kv_lens,
                                    m->cfg.page_size > 0 ? block_table : nullptr, logits, argmax, s);
    e = cudaStreamEndCapture(s, &graph);
    if (le != cudaSuccess) e = le;
    if (e == cudaSuccess) e = cudaGraphInstantiate(&m->gexec, graph, 0);
    if (graph != nullptr) cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail_cuda(m, e, "tq_decode_step_graph: capture");
    m->gkey.batch = batch;
    m->gkey.stream = stream;
    for (int i = 0; i < 6; ++i) m->gkey.p[i] = ptrs[i];
  }
  e = cudaGraphLaunch(m->gexec, s);
  if (e != cudaSuccess) return fail_cuda(m, e, "tq_decode_step_graph: launch");
  return TQ_OK;
}

tq_status tq_model_status(tq_model* m, void* stream, uint32_t* bits) {
  if (m == nullptr || bits == nullptr) return set_error("model and status_bits must not be NULL"), TQ_REFUSED;
  *bits = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  uint32_t v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, m->status(), 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && v != 0) e = cudaMemset(m->status(), 0, 4);
  if (e != cudaSuccess) return fail_cuda(m, e, "tq_model_status");
  *bits = v;
  if (v != 0) {
    set_error("device status 0x%x (%s%s%s); the model is poisoned", v,
              (v & TQ_DEV_BAD_TOKEN) ? "token id out of range " : "",
              (v & TQ_DEV_KV_OVERFLOW) ? "position or cache slot out of range " : "",
              (v & TQ_DEV_WAIT_TIMEOUT) ? "device wait timed out" : "");
    m->poisoned = true;
    m->poison_reason = g_last_error;
    return TQ_INTERNAL;
  }
  return TQ_OK;
}

tq_status tq_model_set_wait_limit(tq_model* m, uint32_t polls) {
  if (refuse_if_poisoned(m)) return TQ_REFUSED;
  if (m->chain_wait_limit != polls && m->gexec != nullptr) {  // a captured step keeps the old value
    cudaGraphExecDestroy(m->gexec);
    m->gexec = nullptr;
  }
  m->chain_wait_limit = polls;
  return TQ_OK;
}

tq_status tq_decode_chain(tq_model* m, int32_t layer, void* stream) {
  if (refuse_if_poisoned(m)) return TQ_REFUSED;
  if (layer < 0 || layer >= m->cfg.n_layers)
    return set_error("layer=%d outside [0, n_layers=%d)", layer, m->cfg.n_layers), TQ_REFUSED;
  const tq::GemvChain ch = layer_chain(m, layer, 1, m->x(), 1, nullptr);
  cudaError_t e = tq::launch_gemv_chain(m->cfg.wtype, ch, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(m, e, "tq_decode_chain");
  return TQ_OK;
}

int tq_model_poisoned(const tq_model* m) { return (m != nullptr && m->poisoned) ? 1 : 0; }

int32_t tq_decode_launches(const tq_model* m, int32_t batch) {
  if (m == nullptr) return 0;
  // batch 1: embed, Q/K/V of layer 0, (attention, chain) per layer, argmax finish;
  // batch >= 2: embed, 9 per layer (4 fragment tables, 4 GEMMs, attention), head table + GEMM + argmax
  return batch >= 2 ? 4 + 9 * m->cfg.n_layers : 3 + 2 * m->cfg.n_layers;
}

void tq_model_free(tq_model* m) {
  if (m == nullptr) return;
  if (m->gexec != nullptr) cudaGraphExecDestroy(m->gexec);
  delete m;
}

// ------------------------------------------------------------- formats --

tq_status tq_qmat_bytes(int32_t wtype, int64_t rows, int64_t cols, int64_t* qs_bytes, int64_t* d_bytes) {
  if (!tiled_wtype(wtype)) return set_error("wtype must be 2, 4 or 8"), TQ_REFUSED;
  if (rows < 0 || cols < 0 || cols % 256 != 0) return set_error("cols must be a multiple of 256"), TQ_REFUSED;
  const int64_t blocks = tq::tiled_rows(rows) * (cols / 32);
  if (qs_bytes != nullptr) *qs_bytes = blocks * (wtype == TQ_Q8_0 ? 32 : 16);
  if (d_bytes != nullptr) *d_bytes = blocks * 2;
  return TQ_OK;
}

tq_status tq_repack(int32_t wtype, const void* blocks, int64_t rows, int64_t cols, void* qs,
                    uint16_t* d, void* stream) {
  if (wtype != TQ_Q4_0 && wtype != TQ_Q8_0)
    return set_error("wtype must be 2 or 8 (affine 4-bit groups: tq_repack_affine4)"), TQ_REFUSED;
  if (rows < 0 || cols < 0 || cols % 256 != 0) return set_error("cols must be a multiple of 256"), TQ_REFUSED;
  if (rows * cols == 0) return TQ_OK;
  if (!blocks || !qs || !d) return set_error("pointers must not be NULL"), TQ_REFUSED;
  if ((reinterpret_cast<uintptr_t>(blocks) & 1u) || !aligned16(qs) || !aligned16(d))
    return set_error("blocks must be 2-byte, qs and d 16-byte aligned"), TQ_REFUSED;
  cudaError_t e = tq::launch_repack(wtype, blocks, rows, cols / 32, qs, d, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_repack");
  return TQ_OK;
}

tq_status tq_quantize(int32_t wtype, const float* w, int64_t rows, int64_t cols, void* blocks, void* stream) {
  if (wtype != TQ_Q4_0 && wtype != TQ_Q8_0)
    return set_error("wtype must be 2 or 8 (affine 4-bit: tq_quantize_affine4)"), TQ_REFUSED;
  if (rows < 0 || cols < 0 || cols % 32 != 0) return set_error("cols must be a multiple of 32"), TQ_REFUSED;
  if (rows * cols == 0) return TQ_OK;
  if (!w || !blocks) return set_error("pointers must not be NULL"), TQ_REFUSED;
  cudaError_t e = tq::launch_quantize(wtype, w, rows * (cols / 32), blocks, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_quantize");
  return TQ_OK;
}

tq_status tq_quantize_affine4(const float* w, int64_t rows, int64_t cols, uint32_t* words, uint16_t* scales,
                              uint16_t* biases, void* stream) {
  if (rows < 0 || cols < 0 || cols % 64 != 0) return set_error("cols must be a multiple of 64"), TQ_REFUSED;
  if (rows * cols == 0) return TQ_OK;
  if (!w || !words || !scales || !biases) return set_error("pointers must not be NULL"), TQ_REFUSED;
  if ((reinterpret_cast<uintptr_t>(w) & 3u) || (reinterpret_cast<uintptr_t>(words) & 3u) ||
      (reinterpret_cast<uintptr_t>(scales) & 1u) || (reinterpret_cast<uintptr_t>(biases) & 1u))
    return set_error("w and words must be 4-byte, scales and biases 2-byte aligned"), TQ_REFUSED;
  cudaError_t e = tq::launch_quantize_affine4(w, rows, cols, words, scales, biases, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_quantize_affine4");
  return TQ_OK;
}

tq_status tq_repack_affine4(const uint32_t* words, const uint16_t* scales, const uint16_t* biases, int64_t rows,
                            int64_t cols, void* qs, uint16_t* d, void* stream) {
  if (rows < 0 || cols < 0 || cols % 256 != 0) return set_error("cols must be a multiple of 256"), TQ_REFUSED;
  if (rows * cols == 0) return TQ_OK;
  if (!words || !scales || !biases || !qs || !d) return set_error("pointers must not be NULL"), TQ_REFUSED;
  if ((reinterpret_cast<uintptr_t>(words) & 3u) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(biases) & 1u) || !aligned16(qs) || !aligned16(d))
    return set_error("words must be 4-byte, scales and biases 2-byte, qs and d 16-byte aligned"), TQ_REFUSED;
  cudaError_t e = tq::launch_repack_affine4(words, scales, biases, rows, cols, qs, d, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_repack_affine4");
  return TQ_OK;
}

tq_status tq_dequantize(int32_t wtype, tq_qmat w, int64_t cols, int64_t row0, int64_t n_rows,
                        float* out, void* stream) {
  if (!tiled_wtype(wtype)) return set_error("wtype must be 2, 4 or 8"), TQ_REFUSED;
  if (cols <= 0 || cols % 256 != 0 || row0 < 0 || n_rows < 0)
    return set_error("cols must be a positive multiple of 256; rows non-negative"), TQ_REFUSED;
  if (n_rows == 0) return TQ_OK;
  if (!w.qs_dev || !w.d_dev || !out) return set_error("pointers must not be NULL"), TQ_REFUSED;
  if (!aligned16(w.qs_dev) || !aligned16(out)) return set_error("qs and out must be 16-byte aligned"), TQ_REFUSED;
  cudaError_t e = tq::launch_dequant(wtype, w.qs_dev, w.d_dev, cols / 32, row0, n_rows, out,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_dequantize");
  return TQ_OK;
}

// ------------------------------------------------------------- ops --

tq_status tq_gemv(int32_t wtype, tq_qmat w, int32_t rows, int32_t cols, const float* x, int32_t batch,
                  const float* residual, float* y, void* stream) {
  if (!tiled_wtype(wtype)) return set_error("wtype must be 2, 4 or 8"), TQ_REFUSED;
  if (rows < 1 || batch < 1 || !tq::gemv_supported(cols))
    return set_error("rows and batch must be >= 1 and cols have a GEMV mapping (got %d)", cols), TQ_REFUSED;
  if (!w.qs_dev || !w.d_dev || !x || !y) return set_error("pointers must not be NULL"), TQ_REFUSED;
  if (!aligned16(w.qs_dev) || !aligned16(w.d_dev) || !aligned16(x))
    return set_error("qs, d and x must be 16-byte aligned"), TQ_REFUSED;
  tq::GemvArgs g{};
  g.seg[0] = seg_of(w, rows);
  g.nseg = 1;
  g.K = cols;
  g.N = rows;
  g.B = batch;
  g.x = x;
  g.y = y;
  g.residual = residual;
  cudaError_t e = tq::launch_gemv(wtype, tq::GEMV_STORE, g, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_gemv");
  return TQ_OK;
}

namespace {
struct GemmScratch {
  size_t x16, inv_s, part, counters, total;
  int64_t part_floats;
};
GemmScratch gemm_scratch(int32_t rows, int32_t n_rows, int32_t cols) {
  GemmScratch g{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  g.x16 = take((size_t)n_rows * cols * 2);
  g.inv_s = take((size_t)n_rows * 4);
  // partial sums of up to 16 splits of K, within the model's cap
  g.part_floats = std::min<int64_t>((int64_t)16 * n_rows * rows, kGemmPartFloats);
  g.part = take((size_t)g.part_floats * 4);
  g.counters = take((size_t)kGemmCounters * 4);
  g.total = off;
  return g;
}
}  // namespace

size_t tq_gemm_scratch_bytes(int32_t rows, int32_t n_rows, int32_t cols) {
  if (rows < 1 || n_rows < 1 || cols < 256 || cols % 256 != 0 || cols > 12288) return 0;
  return gemm_scratch(rows, n_rows, cols).total;
}

tq_status tq_gemm(int32_t wtype, tq_qmat w, int32_t rows, int32_t cols, const float* x, int32_t n_rows,
                  const float* residual, float* y, void* scratch, void* stream) {
  if (!tiled_wtype(wtype)) return set_error("wtype must be 2, 4 or 8"), TQ_REFUSED;
  if (rows < 1 || n_rows < 1 || cols < 256 || cols % 256 != 0 || cols > 12288)
    return set_error("rows, n_rows must be >= 1 and cols a multiple of 256 up to 12288"), TQ_REFUSED;
  if (!w.qs_dev || !w.d_dev || !x || !y || !scratch) return set_error("pointers must not be NULL"), TQ_REFUSED;
  if (!aligned16(w.qs_dev) || !aligned16(w.d_dev) || !aligned16(x) || (residual && !aligned16(residual)) ||
      (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0)
    return set_error("qs, d, x, residual must be 16-byte and scratch 256-byte aligned"), TQ_REFUSED;
  const GemmScratch g = gemm_scratch(rows, n_rows, cols);
  uint8_t* sb = static_cast<uint8_t*>(scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  tq::XPrep16Args p{};
  p.x = x;
  p.ldx = cols;
  p.K = cols;
  p.T = n_rows;
  p.x16 = reinterpret_cast<__half*>(sb + g.x16);
  p.inv_s = reinterpret_cast<float*>(sb + g.inv_s);
  cudaError_t e = cudaMemsetAsync(sb + g.counters, 0, (size_t)kGemmCounters * 4, s);
  if (e == cudaSuccess) e = tq::launch_xprep16(p, s);
  if (e == cudaSuccess) {
    tq::TcGemmArgs q{};
    q.seg[0] = seg_of(w, rows);
    q.nseg = 1;
    q.K = cols;
    q.T = n_rows;
    q.x16 = p.x16;
    q.inv_s = p.inv_s;
    q.y = y;
    q.ldy = rows;
    q.residual = residual;
    q.part = reinterpret_cast<float*>(sb + g.part);
    q.part_cap = g.part_floats;
    q.counters = reinterpret_cast<unsigned*>(sb + g.counters);
    q.n_counters = kGemmCounters;
    e = tq::launch_tcgemm(wtype, q, s);
  }
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_gemm");
  return TQ_OK;
}

tq_status tq_swiglu_gemv(int32_t wtype, tq_qmat gate, tq_qmat up, int32_t ffn, int32_t hidden,
                         const float* x, int32_t batch, const float* gain, float eps, float* out,
                         void* stream) {
  if (!tiled_wtype(wtype)) return set_error("wtype must be 2, 4 or 8"), TQ_REFUSED;
  if (ffn < 1 || batch < 1 || !tq::gemv_supported(hidden))
    return set_error("ffn and batch must be >= 1 and hidden have a GEMV mapping"), TQ_REFUSED;
  if (!gate.qs_dev || !gate.d_dev || !up.qs_dev || !up.d_dev || !x || !out)
    return set_error("pointers must not be NULL"), TQ_REFUSED;
  if (!aligned16(gate.qs_dev) || !aligned16(up.qs_dev) || !aligned16(gate.d_dev) || !aligned16(up.d_dev) ||
      !aligned16(x) || (gain && !aligned16(gain)))
    return set_error("qs, d, x and gain must be 16-byte aligned"), TQ_REFUSED;
  tq::GemvArgs f{};
  f.seg[0] = seg_of(gate, ffn);
  f.seg[1] = seg_of(up, ffn);
  f.nseg = 2;
  f.K = hidden;
  f.N = ffn;
  f.B = batch;
  f.x = x;
  f.gain = gain;
  f.eps = eps;
  f.y = out;
  cudaError_t e = tq::launch_gemv(wtype, tq::GEMV_SWIGLU, f, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_swiglu_gemv");
  return TQ_OK;
}

tq_status tq_sample(const float* logits, int32_t batch, int32_t vocab, const float* temperature,
                    const float* top_p, const float* u, int32_t* out, void* stream) {
  if (batch < 1 || vocab < 1 || vocab > (1 << 24))
    return set_error("batch must be >= 1 and vocab in [1, 2^24]"), TQ_REFUSED;
  if (!logits || !temperature || !top_p || !u || !out) return set_error("pointers must not be NULL"), TQ_REFUSED;
  cudaError_t e = tq::launch_sample(logits, batch, vocab, temperature, top_p, u, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_sample");
  return TQ_OK;
}

tq_status tq_lm_head(int32_t wtype, tq_qmat w, int32_t vocab, int32_t hidden, const float* x,
                     int32_t batch, const float* gain, float eps, float* logits, int32_t* argmax,
                     void* scratch, void* stream) {
  if (!tiled_wtype(wtype)) return set_error("wtype must be 2, 4 or 8"), TQ_REFUSED;
  if (vocab < 1 || batch < 1 || !tq::gemv_supported(hidden))
    return set_error("vocab and batch must be >= 1 and hidden have a GEMV mapping"), TQ_REFUSED;
  if (!w.qs_dev || !w.d_dev || !x || !gain || !argmax || !scratch)
    return set_error("pointers must not be NULL"), TQ_REFUSED;
  if ((reinterpret_cast<uintptr_t>(scratch) & 7u) != 0) return set_error("scratch must be 8-byte aligned"), TQ_REFUSED;
  if (!aligned16(w.qs_dev) || !aligned16(w.d_dev) || !aligned16(x) || !aligned16(gain))
    return set_error("qs, d, x and gain must be 16-byte aligned"), TQ_REFUSED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* keys = static_cast<unsigned long long*>(scratch);
  cudaError_t e = cudaMemsetAsync(keys, 0, batch * sizeof(unsigned long long), s);
  if (e == cudaSuccess) {
    tq::GemvArgs h{};
    h.seg[0] = seg_of(w, vocab);
    h.nseg = 1;
    h.K = hidden;
    h.N = vocab;
    h.B = batch;
    h.x = x;
    h.gain = gain;
    h.eps = eps;
    h.y = logits;
    h.argmax_keys = keys;
    e = tq::launch_gemv(wtype, tq::GEMV_ARGMAX, h, s);
  }
  if (e == cudaSuccess) e = tq::launch_argmax_finish(keys, batch, argmax, s);
  if (e != cudaSuccess) return fail_cuda(nullptr, e, "tq_lm_head");
  return TQ_OK;
}

}  // extern "C"
