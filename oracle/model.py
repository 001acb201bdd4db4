"""Plain forward pass of the Qwen3-style decoder (oracle; test infrastructure).

Every function restates one step of the pages' description, in their order,
with NumPy in float64 (or a caller-chosen dtype).  No blocking, fusion or
reordering beyond the definitions:

* embedding lookup ........ "Всередині LLM ... Qwen3-0.6B на MLX", step 2
* RMSNorm ................. same page, step 3 (eps 1e-6, no mean, no bias)
* RoPE, half-split form ... same page, step 4 (theta 1e6)
* attention with GQA ...... same page, step 5 ("Вся функція уваги"): Q/K/V
  projections, per-head QK-RMSNorm BEFORE RoPE, cache append, KV head h//G
  for query head h, softmax(q k^T / sqrt(hd)) v, causal mask in prefill,
  output projection
* SwiGLU FFN .............. same page, step 6
* pre-norm block .......... same page, step 7
* final norm, LM head ..... same page, step 8; tied to token_embd when the
  model has no output matrix ("Inferencia local y arquitecturas", qwen3.archdef
  epilogue, ``output.weight | token_embd.weight``); only the last position
  ("last(x)") feeds the head
* greedy sampling and the prefill-then-decode loop ... same page, steps 8-9

Sibling architectures ("Inferencia local y arquitecturas", section "El
formato": an architecture is its layer recipe, the same operations in
another order; section "Las operaciones" lists them):

* llama: qwen3 without the per-head Q/K RMSNorm (the qwen3.archdef header
  names that norm as qwen3's only difference from llama);
* qwen2: llama plus three bias additions, read as a bias vector added to the
  q, k and v projections right after their matmuls;
* gemma3-style: the qwen3 recipe with ``gelu_tanh`` (the tanh approximation
  of GELU, which the page distinguishes from exact ``gelu``) as the gate's
  activation, sliding-window attention on a pattern of layers (the one
  ``param`` gemma3 takes), and a final logit softcap (the Gemma 3n
  configuration table of "Alchemize PyTensor ... Gemma 3n": sliding window
  512, final logit softcap 30).  The window counts the query's own position:
  key j is visible to a query at position p iff p - window < j <= p; with
  pattern P, layer i attends the whole context when i % P == P - 1.
  softcap(x) = c * tanh(x / c).

Readings where the pages leave a step open: the mask is
"key position <= query position" (adding -1e9 above the diagonal gives
exactly the same softmax in f64); an f16 KV cache rounds K (after QK-norm and
RoPE) and V to f16 when they are stored; argmax ties go to the lowest index.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import quant


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x * 1/sqrt(mean(x^2) + eps) * g over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x * (1.0 / np.sqrt(ms + eps)) * g


def rope_angles(positions: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """angles[t, i] = pos_t * theta^(-i / (hd/2)) for i < hd/2, in float64."""
    half = head_dim // 2
    freqs = 1.0 / (theta ** (np.arange(half, dtype=np.float64) / half))
    return np.asarray(positions, dtype=np.float64)[:, None] * freqs[None, :]


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Half-split rotation of x [..., T, hd]: pairs (i, i + hd/2) turned by angle[t, i]."""
    hd = x.shape[-1]
    half = hd // 2
    ang = rope_angles(positions, hd, theta)
    cos = np.cos(ang).astype(x.dtype)
    sin = np.sin(ang).astype(x.dtype)
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x1 * sin + x2 * cos], axis=-1)


def softmax(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray, window: int = 0) -> np.ndarray:
    """Grouped-query attention.

    q [nq, T, hd]; k, v [nkv, S, hd] holding key positions 0..S-1;
    q_pos [T] absolute positions of the queries.  Query head h reads KV head
    h // (nq/nkv).  Key j is visible to query t iff j <= q_pos[t] and, with a
    sliding window, j > q_pos[t] - window.
    Returns [nq, T, hd].
    """
    nq, T, hd = q.shape
    nkv, S, _ = k.shape
    G = nq // nkv
    out = np.empty_like(q)
    keys = np.arange(S)[None, :]
    qp = np.asarray(q_pos)[:, None]
    visible = keys <= qp                                                # [T, S]
    if window > 0:
        visible = visible & (keys > qp - window)
    for h in range(nq):
        kv = h // G
        s = (q[h] @ k[kv].T) * (hd ** -0.5)
        s = np.where(visible, s, -np.inf)
        out[h] = softmax(s) @ v[kv]
    return out


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def gelu_tanh(z: np.ndarray) -> np.ndarray:
    """The tanh approximation of GELU: z/2 * (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))."""
    return 0.5 * z * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (z + 0.044715 * z ** 3)))


def softcap(x: np.ndarray, c: float) -> np.ndarray:
    """c * tanh(x / c)."""
    return c * np.tanh(x / c)


class OracleModel:
    """Decoder over quantized block bytes.

    ``weights``: dict mapping GGUF-style names to arrays: block bytes
    [out, in/32, 34|18] for the matrices ``token_embd`` and
    ``blk.{i}.{attn_q,attn_k,attn_v,attn_output,ffn_gate,ffn_up,ffn_down}``
    (optionally ``output``), f32 gains for ``blk.{i}.{attn_norm,ffn_norm,
    attn_q_norm,attn_k_norm}`` (no Q/K norms for llama and qwen2) and
    ``output_norm``, and for qwen2 the f32 biases ``blk.{i}.attn_{q,k,v}_bias``.
    """

    def __init__(self, w, weights: dict, dtype=np.float64, cache_dequant: bool = True):
        self.w = w
        self.weights = weights
        self.dtype = dtype
        self.cache_dequant = cache_dequant
        self._deq: dict = {}

    # -- weights --------------------------------------------------------------
    def matrix(self, name: str) -> np.ndarray:
        if name in self._deq:
            return self._deq[name]
        m = quant.dequantize(self.weights[name], self.w.wtype, self.dtype)
        if self.cache_dequant:
            self._deq[name] = m
        return m

    def gain(self, name: str) -> np.ndarray:
        return np.asarray(self.weights[name], dtype=np.float32).astype(self.dtype)

    def linear(self, x: np.ndarray, name: str) -> np.ndarray:
        """x @ W.T with W stored [out, in]."""
        return x @ self.matrix(name).T

    def head_name(self) -> str:
        return "output" if "output" in self.weights else "token_embd"

    def window_of(self, i: int) -> int:
        """Sliding window of layer i (0: the whole context)."""
        w = self.w
        if w.arch != "gemma3" or w.sliding_window <= 0:
            return 0
        P = w.sliding_pattern
        return 0 if P > 0 and i % P == P - 1 else w.sliding_window

    # -- steps ----------------------------------------------------------------
    def embed(self, tokens) -> np.ndarray:
        blocks = self.weights["token_embd"][np.asarray(tokens, dtype=np.int64)]
        return quant.dequantize(blocks, self.w.wtype, self.dtype)

    def store_kv(self, t: np.ndarray) -> np.ndarray:
        if self.w.kv == "f16":
            return t.astype(np.float16).astype(self.dtype)
        return t

    def attn_block(self, i: int, h: np.ndarray, cache: list, positions: np.ndarray):
        w = self.w
        p = f"blk.{i}"
        T = h.shape[0]
        q = self.linear(h, f"{p}.attn_q").reshape(T, w.n_heads, w.head_dim).transpose(1, 0, 2)
        k = self.linear(h, f"{p}.attn_k").reshape(T, w.n_kv_heads, w.head_dim).transpose(1, 0, 2)
        v = self.linear(h, f"{p}.attn_v").reshape(T, w.n_kv_heads, w.head_dim).transpose(1, 0, 2)
        if w.arch == "qwen2":
            q = q + self.gain(f"{p}.attn_q_bias").reshape(w.n_heads, 1, w.head_dim)
            k = k + self.gain(f"{p}.attn_k_bias").reshape(w.n_kv_heads, 1, w.head_dim)
            v = v + self.gain(f"{p}.attn_v_bias").reshape(w.n_kv_heads, 1, w.head_dim)
        if w.arch in ("qwen3", "gemma3"):
            q = rms_norm(q, self.gain(f"{p}.attn_q_norm"), w.rms_eps)
            k = rms_norm(k, self.gain(f"{p}.attn_k_norm"), w.rms_eps)
        q = rope(q, positions, w.rope_theta)
        k = rope(k, positions, w.rope_theta)
        k = self.store_kv(k)
        v = self.store_kv(v)
        if cache[i] is not None:
            ck, cv = cache[i]
            k = np.concatenate([ck, k], axis=1)
            v = np.concatenate([cv, v], axis=1)
        cache[i] = (k, v)
        o = attention(q, k, v, positions, self.window_of(i))
        o = o.transpose(1, 0, 2).reshape(T, w.n_heads * w.head_dim)
        return self.linear(o, f"{p}.attn_output")

    def ffn_block(self, i: int, h: np.ndarray) -> np.ndarray:
        p = f"blk.{i}"
        gate = self.linear(h, f"{p}.ffn_gate")
        up = self.linear(h, f"{p}.ffn_up")
        act = gelu_tanh(gate) if self.w.arch == "gemma3" else silu(gate)
        return self.linear(act * up, f"{p}.ffn_down")

    def block(self, i: int, x: np.ndarray, cache: list, positions: np.ndarray) -> np.ndarray:
        p = f"blk.{i}"
        h = rms_norm(x, self.gain(f"{p}.attn_norm"), self.w.rms_eps)
        x = x + self.attn_block(i, h, cache, positions)
        h = rms_norm(x, self.gain(f"{p}.ffn_norm"), self.w.rms_eps)
        return x + self.ffn_block(i, h)

    def head(self, x_last: np.ndarray) -> np.ndarray:
        x = rms_norm(x_last, self.gain("output_norm"), self.w.rms_eps)
        logits = self.linear(x, self.head_name())
        if self.w.arch == "gemma3" and self.w.logit_softcap > 0:
            logits = softcap(logits, self.w.logit_softcap)
        return logits

    def new_cache(self) -> list:
        return [None] * self.w.n_layers

    def forward(self, tokens, cache: list, start_pos: int) -> np.ndarray:
        """Run ``tokens`` at positions start_pos.. through every layer, append
        their K/V to ``cache``, and return the logits of the last position."""
        tokens = np.asarray(tokens)
        positions = np.arange(start_pos, start_pos + len(tokens))
        x = self.embed(tokens)
        for i in range(self.w.n_layers):
            x = self.block(i, x, cache, positions)
        return self.head(x[-1])

    def forward_nocache(self, tokens) -> np.ndarray:
        """Full-prefix recomputation with no carried state: logits of the last token."""
        return self.forward(tokens, self.new_cache(), 0)


def argmax(logits: np.ndarray) -> int:
    """Greedy choice; np.argmax returns the first (lowest-index) maximum."""
    return int(np.argmax(logits))


def run_greedy(model: OracleModel, prompt, n_steps: int, teacher: Optional[list] = None):
    """Prefill ``prompt`` then ``n_steps`` single-token decode steps.

    Decode step s feeds token t_s at position len(prompt) + s, where t_0 is
    the prefill's argmax and t_{s+1} the argmax of step s -- or, with teacher
    forcing, ``teacher[s]``.  Returns (tokens t_0..t_n_steps, logits list of
    n_steps + 1 arrays: the prefill's and each step's).
    """
    cache = model.new_cache()
    P = len(prompt)
    logits = [model.forward(prompt, cache, 0)]
    toks = [argmax(logits[0])]
    for s in range(n_steps):
        feed = toks[s] if teacher is None else int(teacher[s])
        logits.append(model.forward([feed], cache, P + s))
        toks.append(argmax(logits[-1]))
    return toks, logits


def synth_weights(w) -> dict:
    """Quantized weights of workload ``w`` from the seeded generator, quantized
    by this oracle's own encoder."""
    import synth
    out = {}
    for name in w.matrices():
        out[name] = quant.quantize(synth.host_tensor(w, name), w.wtype)
    for name in w.gains() + w.biases():
        out[name] = synth.host_tensor(w, name)
    return out
