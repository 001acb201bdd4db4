/* tq -- decode step of a Qwen3-style decoder over Q8_0 / Q4_0 block-quantized
 * weights, on one NVIDIA GB300 (sm_103a).  C ABI of libtq.so.
 *
 * What is computed is the forward pass of the pages "Всередині LLM: чисте
 * виконання на Python для Qwen3-0.6B на MLX" (steps 2-9: embedding, RMSNorm,
 * RoPE, grouped-query attention with a KV cache, SwiGLU, pre-norm block, LM
 * head and greedy sampling, prefill then one token per step) and
 * "Inferencia local y arquitecturas" (section "El formato": the qwen3.archdef
 * layer graph, per-head QK-RMSNorm before RoPE, tied LM head
 * output.weight | token_embd.weight, last(x) before the head; section "Elegir
 * el motor": weights stay quantized and are multiplied in f32 with no
 * activation quantization).  Handle, status and poisoning conventions follow
 * the tessl_torch README, sections "Handle ownership, closing and errors" and
 * "How the buffers cross".
 *
 * Conventions for every call:
 *  - All memory is the caller's.  Pointers named *_dev are device pointers,
 *    all others host pointers.  The library allocates no device memory; a
 *    model keeps the pointers it was given, which must stay valid until
 *    tq_model_free().
 *  - Work is enqueued on the caller's CUDA stream (NULL = legacy default
 *    stream) and the call returns without waiting for the GPU, except where
 *    a call says it synchronizes.
 *  - Return status: TQ_OK; TQ_REFUSED (an argument is invalid: nothing was
 *    enqueued, the model stays usable); TQ_INTERNAL (a CUDA error: the model
 *    is poisoned and refuses every later call with TQ_REFUSED; free it and
 *    create a new one, keeping every buffer it was given alive until the
 *    free).  tq_last_error() describes the last failure on the calling thread.
 *  - Weight matrices are [out][in] with blocks of 32 along `in`, in the tiled
 *    layout made by tq_repack() (tq_qmat).
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TQ_API __attribute__((visibility("default")))
#else
#define TQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { TQ_OK = 0, TQ_REFUSED = 1, TQ_INTERNAL = 2 } tq_status;

/* Block formats (GGUF type ids).  Q8_0: 32 weights, fp16 d, int8 q; value
 * d*q.  Q4_0: 32 weights, fp16 d, 4-bit q; value d*(q-8).  GGUF byte order of
 * one block: Q8_0 = fp16 d, int8 q[32] (34 B); Q4_0 = fp16 d, uint8 qs[16],
 * qs[j] = q[j] | q[j+16] << 4 (18 B).
 * AFFINE4 ("Alchemize PyTensor ... Gemma 3n", the affine-4 checkpoint):
 * groups of 64 inputs, 4-bit q, bf16 scale s and bias b per group; value
 * q*s + b.  Its source layout is MLX's planar one: words [rows][cols/8]
 * uint32 (input c in bits 4(c%8) .. 4(c%8)+3 of word c/8), scales and biases
 * [rows][cols/64] bf16 (tq_quantize_affine4, tq_repack_affine4). */
typedef enum { TQ_Q4_0 = 2, TQ_AFFINE4 = 4, TQ_Q8_0 = 8 } tq_wtype;
typedef enum { TQ_KV_F32 = 0, TQ_KV_F16 = 1 } tq_kvtype;

/* Bits of the device status word (tq_model_status()). */
enum {
  TQ_DEV_BAD_TOKEN = 1u,     /* a token id >= vocab: its embedding was read as zeros */
  TQ_DEV_KV_OVERFLOW = 2u,   /* a position or cache slot >= capacity: the write was skipped */
  TQ_DEV_WAIT_TIMEOUT = 4u   /* a bounded device-side wait gave up */
};

/* Model shape and capacity.  Sizes must satisfy: head_dim in {64, 128};
 * n_heads % n_kv_heads == 0 with n_heads / n_kv_heads <= 8; hidden, ffn and
 * n_heads*head_dim multiples of 256 and at most 12288; max_batch >= 1.
 * KV cache: page_size == 0 selects the contiguous layout
 *   [n_layers][max_batch][n_kv_heads][max_ctx][head_dim]
 * (sequence b of a decode batch uses slot b); page_size > 0 (a multiple of
 * 32) selects the paged layout [n_layers][n_pages][n_kv_heads][page_size][head_dim]
 * addressed through a block table [batch][max_ctx / page_size]. */
typedef struct {
  int32_t vocab, hidden, n_layers, n_heads, n_kv_heads, head_dim, ffn;
  float rms_eps, rope_theta;
  int32_t wtype;        /* tq_wtype */
  int32_t kvtype;       /* tq_kvtype */
  int32_t max_batch;    /* sequences in one decode step */
  int32_t max_ctx;      /* tokens a sequence may hold (positions 0 .. max_ctx-1) */
  int32_t max_prefill;  /* tokens one tq_prefill call may process */
  int32_t page_size;    /* 0 = contiguous cache */
  int32_t n_pages;      /* pages in the pool (paged cache only) */
  /* Layer recipe ("Inferencia local y arquitecturas", sections "El formato"
   * and "Las operaciones": an architecture is the same operations in another
   * order).  All zero = qwen3. */
  int32_t arch;            /* tq_arch */
  int32_t sliding_window;  /* gemma3: a sliding layer's query at cache index p sees keys j with
                              p - sliding_window < j <= p (0 = every layer sees the whole context) */
  int32_t sliding_pattern; /* gemma3: layer l sees the whole context when l % p == p - 1
                              (0 = every layer slides) */
  float logit_softcap;     /* gemma3: logits = c * tanh(logits / c) (0 = none) */
} tq_config;

/* qwen3: per-head RMSNorm of q and k before RoPE, SiLU-gated FFN;
 * llama: qwen3 without the per-head norm (attn_q_norm / attn_k_norm unused);
 * qwen2: llama plus bias vectors added to q, k and v after their matmuls;
 * gemma3: qwen3 with a tanh-approximated-GELU gate, sliding-window attention
 *         on a layer pattern and a final logit softcap (the config fields above). */
typedef enum { TQ_ARCH_QWEN3 = 0, TQ_ARCH_LLAMA = 1, TQ_ARCH_QWEN2 = 2, TQ_ARCH_GEMMA3 = 3 } tq_arch;

/* One quantized matrix [rows][cols] (cols a multiple of 256) in the tiled
 * layout.  Rows are padded with zero rows to a multiple of 16 (R rows) and
 * grouped in tiles of 16; the 8-block runs of a tile row ("units", 16 rows x
 * 256 inputs) are stored tile after tile:
 *  qs_dev: R/16 * cols/256 units of 2048 (Q4_0, AFFINE4) or 4096 (Q8_0) bytes,
 *          i.e. R * cols/32 * 16 (Q4_0, AFFINE4) or * 32 (Q8_0) bytes in all;
 *  d_dev:  R/16 * cols/256 units of 128 fp16 scales (R * cols/32 scales).
 * Inside a unit, 32-bit code word i (Q4_0: bytes 4i..4i+3 of the block's 16
 * nibble bytes, i < 4; Q8_0: codes 4i..4i+3, i < 8) of block j (0-7) of tile
 * row rr = 8h + g lies at byte
 *   Q4_0: ((h*2 + j/4)*32 + 4g + i)*16 + (j%4)*4
 *   Q8_0: ((h*4 + j/2)*32 + 4g + i%4)*16 + (j%2)*8 + (i/4)*4
 * and its scale at element (h*8 + g)*8 + j; so each lane of a warp loads the
 * words of its tensor-core operand fragment with one 16-byte load.
 * AFFINE4 takes the Q4_0 arrangement (each 32-input block's codes as a Q4_0
 * block's bytes q[j] | q[j+16] << 4); its 16-bit elements hold the bf16
 * scale of group k (blocks 2k, 2k+1) at block 2k and its bias at block 2k+1.
 * tq_qmat_bytes() gives the sizes.  Both pointers 16-byte aligned. */
typedef struct {
  const void* qs_dev;
  const uint16_t* d_dev;
} tq_qmat;

typedef struct {
  tq_qmat attn_q, attn_k, attn_v, attn_output, ffn_gate, ffn_up, ffn_down;
  const float* attn_norm_dev;     /* [hidden] */
  const float* ffn_norm_dev;      /* [hidden] */
  const float* attn_q_norm_dev;   /* [head_dim] (qwen3, gemma3; else unused) */
  const float* attn_k_norm_dev;   /* [head_dim] (qwen3, gemma3; else unused) */
  const float* attn_q_bias_dev;   /* qwen2: [n_heads * head_dim]; else unused */
  const float* attn_k_bias_dev;   /* qwen2: [n_kv_heads * head_dim] */
  const float* attn_v_bias_dev;   /* qwen2: [n_kv_heads * head_dim] */
} tq_layer;

typedef struct {
  tq_qmat token_embd;             /* [vocab][hidden] */
  tq_qmat output;                 /* [vocab][hidden]; qs_dev == NULL: tied to token_embd */
  const float* output_norm_dev;   /* [hidden] */
  const tq_layer* layers;         /* host array of n_layers, copied by tq_model_create */
} tq_weights;

typedef struct tq_model tq_model;

/* ---------------------------------------------------------------- model -- */

/* Device workspace bytes a model of this configuration needs (activations,
 * attention partials, RoPE table, status word).  0 if the configuration is
 * invalid (tq_last_error() says why). */
TQ_API size_t tq_workspace_bytes(const tq_config* cfg);

/* Bytes of one KV cache buffer (K or V) for this configuration. */
TQ_API size_t tq_kv_cache_bytes(const tq_config* cfg);

/* Create a model over caller-owned device memory: the weights, a workspace
 * of tq_workspace_bytes() (256-byte aligned) and the K and V caches of
 * tq_kv_cache_bytes() each.  Synchronizes the device once (it uploads the
 * RoPE table, computed on the host in double precision, and clears the
 * workspace).  The cache contents are not touched. */
TQ_API tq_status tq_model_create(const tq_config* cfg, const tq_weights* weights, void* workspace_dev,
                          void* k_cache_dev, void* v_cache_dev, tq_model** out);

/* Prefill: run n_tokens tokens of one sequence at positions
 * start_pos .. start_pos+n_tokens-1 (causal attention over the sequence's
 * cached positions 0 .. start_pos-1 and the new ones), store their K/V, and
 * produce the last position's logits and greedy token.
 *  seq:             cache slot (contiguous cache), 0 <= seq < max_batch;
 *                   ignored for a paged cache;
 *  tokens_dev:      [n_tokens] int32 token ids;
 *  block_table_dev: paged cache only: [max_ctx / page_size] int32 page ids of
 *                   this sequence (NULL for a contiguous cache);
 *  logits_dev:      [vocab] f32, or NULL;
 *  argmax_dev:      [1] int32, the lowest index of the largest logit.
 * Refused when n_tokens < 1, n_tokens > max_prefill or
 * start_pos + n_tokens > max_ctx. */
TQ_API tq_status tq_prefill(tq_model* m, int32_t seq, const int32_t* tokens_dev, int32_t n_tokens,
                     int32_t start_pos, const int32_t* block_table_dev, float* logits_dev,
                     int32_t* argmax_dev, void* stream);

/* One decode step for `batch` sequences: sequence b feeds tokens_dev[b] at
 * position positions_dev[b], appends its K/V at cache index kv_lens_dev[b]
 * and attends over indices 0 .. kv_lens_dev[b] (kv_lens_dev[b] + 1 keys).
 *  tokens_dev, positions_dev, kv_lens_dev: [batch] int32;
 *  block_table_dev: paged cache: [batch][max_ctx / page_size] int32, else NULL;
 *  logits_dev: [batch][vocab] f32, or NULL;
 *  argmax_dev: [batch] int32.
 * Refused when batch < 1 or batch > max_batch.  Device-side range errors
 * (token >= vocab, kv_lens + 1 > max_ctx) set bits of the status word. */
TQ_API tq_status tq_decode_step(tq_model* m, int32_t batch, const int32_t* tokens_dev,
                         const int32_t* positions_dev, const int32_t* kv_lens_dev,
                         const int32_t* block_table_dev, float* logits_dev, int32_t* argmax_dev,
                         void* stream);

/* One step of continuous batching: n_rows token rows from n_seq sequences
 * at once, any mix of prompt chunks (several rows of one sequence) and
 * decode tokens (one row), through every layer with the projections as GEMMs
 * over all rows ("Всередині LLM ... Qwen3-0.6B на MLX", step 9: a prompt pass
 * and single-token steps are the same forward pass over different rows;
 * "PyTensor Beyond PyMC", section "What the current speed tells us": paged
 * cache and continuous batching).  Row t is token tokens_dev[t] of the
 * sequence in block-table row (paged cache: block_table_dev is
 * [max_batch][max_ctx / page_size]) or cache slot (contiguous)
 * row_seq_dev[t] in [0, max_batch), at position and cache index
 * row_pos_dev[t]; it appends its K/V there and attends over indices
 * 0 .. row_pos_dev[t] of its sequence.  Where rows t0 .. t0 + 128/G - 1 (t0 a
 * multiple of 128/G, G query heads per KV head) are consecutive positions of
 * one sequence, an f16 cache's attention runs them as one flash-attention
 * block, as in tq_prefill; other rows attend one by one.  A
 * sequence's rows must come in ascending position order with no gaps after
 * what its cache already holds.  For each sequence b < n_seq, last_row_dev[b]
 * is the row whose logits / greedy token are produced:
 *  logits_dev: [n_seq][vocab] f32, or NULL (then n_seq > 1 needs max_batch > 1);
 *  argmax_dev: [n_seq] int32.
 * Admission and eviction are the caller's: a sequence's pages are its
 * block-table row; freeing them (and reusing them for a new sequence, which
 * overwrites from position 0) is bookkeeping on the host.  Refused when
 * n_rows < 1 or > max_prefill, n_seq < 1 or > max_batch or > n_rows.
 * Device-side range errors (a bad token, sequence index, position, page or
 * last row) set status bits and skip the access. */
TQ_API tq_status tq_step(tq_model* m, int32_t n_rows, const int32_t* tokens_dev, const int32_t* row_seq_dev,
                         const int32_t* row_pos_dev, int32_t n_seq, const int32_t* last_row_dev,
                         const int32_t* block_table_dev, float* logits_dev, int32_t* argmax_dev, void* stream);

/* Capture tq_decode_step(batch, ...) with these exact pointers into a CUDA
 * graph owned by the model and replay it on `stream`: same results, fewer
 * launch gaps.  The graph is rebuilt when any argument changes. */
TQ_API tq_status tq_decode_step_graph(tq_model* m, int32_t batch, const int32_t* tokens_dev,
                               const int32_t* positions_dev, const int32_t* kv_lens_dev,
                               const int32_t* block_table_dev, float* logits_dev,
                               int32_t* argmax_dev, void* stream);

/* Wait for `stream`, then read and clear the device status word into
 * *status_bits.  A non-zero word poisons the model and returns TQ_INTERNAL. */
TQ_API tq_status tq_model_status(tq_model* m, void* stream, uint32_t* status_bits);

/* Polls after which each grid-wide wait between the phases of the decode
 * GEMV chains gives up (0 restores the default of 2^24 polls, far longer than
 * any step).  A wait that gives up sets TQ_DEV_WAIT_TIMEOUT in the status
 * word, and the launch runs on without waiting (no wait is left unbounded
 * and every bulk copy it issued lands before it exits), so its results are
 * meaningless; tq_model_status() then reports the bit and poisons the model.
 * For tests of that failure path: a limit of one or two polls is shorter than
 * the CTAs of a chain take to meet.  Applies to steps enqueued afterwards (a
 * captured decode graph is dropped and re-captured).  The tessl_torch README,
 * "Handle ownership, closing and errors", sets the rule that a failed wait
 * poisons the handle rather than hanging. */
TQ_API tq_status tq_model_set_wait_limit(tq_model* m, uint32_t polls);

/* 1 if the model is poisoned (a CUDA error or a device status bit was seen). */
TQ_API int tq_model_poisoned(const tq_model* m);

/* One step of the batch-1 decode path on its own: the GEMV chain that
 * follows layer `layer`'s attention ("Всередині LLM ... Qwen3-0.6B на MLX",
 * steps 5-7: output projection + residual, RMSNorm + SwiGLU FFN + residual,
 * then the next layer's RMSNorm + Q/K/V projections, or after the last layer
 * step 8's final norm + LM head + argmax keys), exactly as tq_decode_step
 * launches it, over the workspace's current activations.  For measuring the
 * chain inside the step's launch configuration; the workspace's activations
 * are overwritten.  Refused when layer is outside [0, n_layers). */
TQ_API tq_status tq_decode_chain(tq_model* m, int32_t layer, void* stream);

/* Number of kernel launches one tq_decode_step(batch) enqueues. */
TQ_API int32_t tq_decode_launches(const tq_model* m, int32_t batch);

/* Release the model object (not the caller's memory).  NULL is ignored. */
TQ_API void tq_model_free(tq_model* m);

/* Description of the last failure on the calling thread ("" if none). */
TQ_API const char* tq_last_error(void);

/* ------------------------------------------------------- weight formats -- */

/* Bytes of the qs and d arrays of a [rows][cols] matrix in the tiled layout
 * (tq_qmat).  Refused when cols % 256 != 0 or a size is negative. */
TQ_API tq_status tq_qmat_bytes(int32_t wtype, int64_t rows, int64_t cols, int64_t* qs_bytes,
                               int64_t* d_bytes);

/* GGUF-order blocks -> tiled layout (tq_qmat), padding rows included.
 *  blocks_dev: [rows][cols/32] blocks of 34 (Q8_0) or 18 (Q4_0) bytes;
 *  qs_dev, d_dev: outputs as described for tq_qmat.
 * A matrix may be repacked in row chunks whose first row is a multiple of
 * 16, with qs_dev/d_dev advanced by that many rows' bytes.
 * Refused when cols % 256 != 0 or a pointer is NULL or misaligned. */
TQ_API tq_status tq_repack(int32_t wtype, const void* blocks_dev, int64_t rows, int64_t cols,
                    void* qs_dev, uint16_t* d_dev, void* stream);

/* Encode f32 weights [rows][cols] into GGUF-order Q8_0 / Q4_0 blocks
 * (Q8_0: d = max|w|/127; Q4_0: d = m/-8 with m the first weight of largest
 * magnitude, with its sign; q = round-half-away(w/d) in f32, clamped to
 * [-127,127] or, plus 8, to [0,15]; the stored scale is fp16(d), round to
 * nearest even; an all-zero block gets d = 0). */
TQ_API tq_status tq_quantize(int32_t wtype, const float* w_dev, int64_t rows, int64_t cols,
                      void* blocks_dev, void* stream);

/* Encode f32 weights [rows][cols] (cols a multiple of 64) into MLX-layout
 * affine 4-bit groups: per group of 64 inputs of a row, s = (max - min) / 15
 * and b = min in f32, q = round-half-away((w - b) / s) in f32 clamped to
 * [0, 15] (q = 0 when s = 0); the stored s and b are bf16, rounded to
 * nearest even.  words_dev [rows][cols/8] uint32, scales_dev and
 * biases_dev [rows][cols/64] bf16 bit patterns. */
TQ_API tq_status tq_quantize_affine4(const float* w_dev, int64_t rows, int64_t cols, uint32_t* words_dev,
                                     uint16_t* scales_dev, uint16_t* biases_dev, void* stream);

/* MLX-layout affine 4-bit groups (as written by tq_quantize_affine4) ->
 * tiled layout (tq_qmat of wtype TQ_AFFINE4), padding rows included; row
 * chunks as for tq_repack.  Refused when cols % 256 != 0 or a pointer is
 * NULL or misaligned. */
TQ_API tq_status tq_repack_affine4(const uint32_t* words_dev, const uint16_t* scales_dev,
                                   const uint16_t* biases_dev, int64_t rows, int64_t cols, void* qs_dev,
                                   uint16_t* d_dev, void* stream);

/* Decode rows [row0, row0+n_rows) of a tiled matrix to f32 (exact for Q8_0
 * and Q4_0; AFFINE4: q*s + b rounded once to f32). */
TQ_API tq_status tq_dequantize(int32_t wtype, tq_qmat w, int64_t cols, int64_t row0, int64_t n_rows,
                        float* out_dev, void* stream);

/* ----------------------------------------------------------- single ops -- */

/* y[b][r] = (residual ? residual[b][r] : 0) + sum_c W[r][c] * x[b][c], for
 * b < batch, r < rows: the decode GEMV on its own (x, y, residual: f32,
 * row-major with leading dimensions cols and rows; residual may alias y). */
TQ_API tq_status tq_gemv(int32_t wtype, tq_qmat w, int32_t rows, int32_t cols, const float* x_dev,
                  int32_t batch, const float* residual_dev, float* y_dev, void* stream);

/* Bytes of scratch tq_gemm needs for a [rows][cols] matrix and n_rows rows
 * of input (0 when the sizes are invalid): the fp16 input rows, their scales,
 * split-K partial sums and split counters. */
TQ_API size_t tq_gemm_scratch_bytes(int32_t rows, int32_t n_rows, int32_t cols);

/* The GEMM of prefill and batched decode on its own ("Всередині LLM ...
 * Qwen3-0.6B на MLX", step 9: the prompt's positions through the same
 * projections): y[t][r] = (residual ? residual[t][r] : 0) +
 * sum_c W[r][c] * x[t][c] for t < n_rows, r < rows, on the tcgen05 tensor
 * cores: the weights decoded to fp16 in shared memory (d * (q - 8) or d * q
 * rounded once), each row of x scaled by a power of two and rounded to fp16,
 * products summed in f32, so |error| <= about 2^-10 * sum_c |W[r][c] x[t][c]|;
 * each weight tile is decoded once per 256 rows of x (x, y, residual: f32
 * row-major with leading dimensions cols and rows; residual may alias y; all
 * 16-byte aligned).  With few rows of x, K is split across CTAs as in the
 * model's batched decode (the partial sums are added in split order).
 * scratch_dev: at least tq_gemm_scratch_bytes(rows, n_rows, cols) bytes of
 * device memory, 256-byte aligned, owned by the caller; the call must not
 * overlap another use of it.  Refused
 * when cols % 256 != 0 or cols > 12288, a size is < 1 or a pointer NULL or
 * misaligned. */
TQ_API tq_status tq_gemm(int32_t wtype, tq_qmat w, int32_t rows, int32_t cols, const float* x_dev,
                         int32_t n_rows, const float* residual_dev, float* y_dev, void* scratch_dev,
                         void* stream);

/* RMSNorm + gate/up projections + SwiGLU on their own ("Всередині LLM ...
 * Qwen3-0.6B на MLX", steps 3 and 6): out[b][i] = silu(g_i) * u_i with
 * g = Wg h, u = Wu h, h = rms_norm(x[b], gain) (gain NULL: h = x[b]).
 * x_dev [batch][hidden], out_dev [batch][ffn], f32. */
TQ_API tq_status tq_swiglu_gemv(int32_t wtype, tq_qmat gate, tq_qmat up, int32_t ffn, int32_t hidden,
                                const float* x_dev, int32_t batch, const float* gain_dev, float eps,
                                float* out_dev, void* stream);

/* Greedy head on its own ("Всередині LLM ... Qwen3-0.6B на MLX", step 8):
 * logits[b] = W * rms_norm(x[b], gain) and argmax[b] = the lowest index of the
 * largest logit.  logits_dev may be NULL; scratch_dev holds 8*batch bytes
 * (8-byte aligned) of per-row argmax keys. */
TQ_API tq_status tq_lm_head(int32_t wtype, tq_qmat w, int32_t vocab, int32_t hidden,
                     const float* x_dev, int32_t batch, const float* gain_dev, float eps,
                     float* logits_dev, int32_t* argmax_dev, void* scratch_dev, void* stream);

/* Temperature / top-p sampling ("Всередині LLM ... Qwen3-0.6B на MLX", step
 * 8, sample(logits, temperature, top_p)), on the device, one token per row:
 *  logits_dev:      [batch][vocab] f32 (for instance tq_decode_step's logits);
 *  temperature_dev: [batch] f32; 0 selects greedy decoding (the lowest index
 *                   of the largest logit), > 0 divides the logits before the
 *                   softmax;
 *  top_p_dev:       [batch] f32: the tokens, ordered by descending probability
 *                   (equal probabilities by ascending index), are kept up to
 *                   and including the first whose cumulative probability
 *                   reaches top_p, and renormalised;
 *  u_dev:           [batch] f32 uniform numbers in [0, 1): the drawn token is
 *                   the first kept token whose cumulative renormalised
 *                   probability exceeds u (the caller owns the randomness);
 *  out_dev:         [batch] int32 token ids.
 * Each unnormalised probability is an f32 exp2 of (l - max) log2(e) / T,
 * held as an integer multiple of 2^-(62 - ceil(log2 vocab)) of the largest,
 * and the cumulative sums are exact integer sums (the same token for the
 * same inputs, whatever the timing); a draw whose u lies within the f32
 * exp's rounding of a cumulative sum may fall on the neighbouring token.  A
 * row whose largest logit is +inf is decoded greedily; a NaN top_p keeps
 * every token, a NaN u reads as 0.  Refused when
 * batch < 1, vocab < 1 or vocab > 2^24, or a pointer is NULL. */
TQ_API tq_status tq_sample(const float* logits_dev, int32_t batch, int32_t vocab, const float* temperature_dev,
                           const float* top_p_dev, const float* u_dev, int32_t* out_dev, void* stream);

/* ------------------------------------------------- allocation-free head -- */

/* Largest batch of one tq_lm_head_static() call. */
#define TQ_LM_HEAD_STATIC_MAX_BATCH 4096

/* tq_lm_head() without the caller's scratch, for callers that cannot
 * allocate device memory (a plugin inside a host framework that owns the
 * device memory pool; a thread that must not risk the device-wide
 * synchronization of cudaMalloc).  The pages have no counterpart: this is an
 * integration entry point.  The argmax keys live in a static device array of
 * TQ_LM_HEAD_STATIC_MAX_BATCH * 8 bytes (held by every GPU that loads the
 * library until exit); batch above that maximum is refused (TQ_REFUSED).  The
 * array is shared by all calls and keeps the last call's contents; each call
 * clears the rows it uses.  Calls whose GPU work overlaps race on the array:
 * serialize them.  The first call on a device looks the array up with that
 * device current; make it before any stream capture.  The looked-up address is
 * kept for the life of the process: after cudaDeviceReset() on that device it
 * is stale, so do not call this entry point on a device that was reset.  Nothing is allocated
 * (no cudaMalloc/cudaFree, no allocating library routine).  Other arguments
 * and results are those of tq_lm_head(). */
TQ_API tq_status tq_lm_head_static(int32_t wtype, tq_qmat w, int32_t vocab, int32_t hidden,
                                   const float* x_dev, int32_t batch, const float* gain_dev,
                                   float eps, float* logits_dev, int32_t* argmax_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
