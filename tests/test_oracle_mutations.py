"""Planted mistakes in the oracle (on the CPU, via monkeypatch) must be caught
by the pins: evidence that the pins constrain what they claim to."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import model as om
from oracle import quant
import test_oracle_pins as pins


def _wrong_gqa(q, k, v, q_pos):
    nq, T, hd = q.shape
    nkv = k.shape[0]
    out = np.empty_like(q)
    vis = np.arange(k.shape[1])[None, :] <= np.asarray(q_pos)[:, None]
    for h in range(nq):
        kv = h % nkv                                     # planted: modulo head map
        s = np.where(vis, (q[h] @ k[kv].T) / math.sqrt(hd), -np.inf)
        out[h] = om.softmax(s) @ v[kv]
    return out


def _interleaved_rope(x, positions, theta):
    hd = x.shape[-1]
    ang = om.rope_angles(positions, hd, theta)
    c, s = np.cos(ang), np.sin(ang)
    y = x.copy()
    y[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s  # planted: adjacent pairs
    y[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return y


def test_planted_gqa_map_is_caught(monkeypatch):
    monkeypatch.setattr(om, "attention", _wrong_gqa)
    with pytest.raises(AssertionError):
        pins.test_attention_prefill_matches_sdpa(8, 2)


def test_planted_interleaved_rope_is_caught(monkeypatch):
    monkeypatch.setattr(om, "rope", _interleaved_rope)
    with pytest.raises(AssertionError):
        pins.test_rope_closed_form_pairs_and_frequencies()
    with pytest.raises(AssertionError):
        pins.test_rope_equals_complex_rotation()


def test_planted_norm_after_rope_is_caught(monkeypatch):
    orig = om.OracleModel.attn_block

    def swapped(self, i, h, cache, positions):
        real_rope, real_norm = om.rope, om.rms_norm
        calls = {"n": 0}

        def rope_then_norm(x, pos, theta):
            return x                                    # rope deferred ...

        def norm_then_rope(x, g, eps):
            y = real_norm(x, g, eps)
            if x.ndim == 3:                             # per-head norm: apply rope first
                y = real_norm(real_rope(x, positions, self.w.rope_theta), g, eps)
            return y
        monkeypatch.setattr(om, "rope", rope_then_norm)
        monkeypatch.setattr(om, "rms_norm", norm_then_rope)
        try:
            return orig(self, i, h, cache, positions)
        finally:
            monkeypatch.setattr(om, "rope", real_rope)
            monkeypatch.setattr(om, "rms_norm", real_norm)

    monkeypatch.setattr(om.OracleModel, "attn_block", swapped)
    with pytest.raises(AssertionError):
        pins.test_model_matches_torch_library_composition()


def test_planted_half_even_rounding_is_caught(monkeypatch):
    monkeypatch.setattr(quant, "round_half_away", lambda x: np.round(x))
    with pytest.raises(AssertionError):
        pins.test_hand_worked_block("q4_0_block.txt", "q4_0")
    with pytest.raises(AssertionError):
        pins.test_hand_worked_block("q8_0_block.txt", "q8_0")


def test_planted_unsigned_q4_extreme_is_caught(monkeypatch):
    real = quant.quantize_q4_0

    def unsigned(w):
        w = np.asarray(w, np.float32)
        b = w.reshape(-1, 32)
        flip = b[np.arange(b.shape[0]), np.argmax(np.abs(b), 1)] < 0
        b = np.where(flip[:, None], -b, b)              # planted: extreme always positive
        out = real(b)
        return out.reshape(*w.shape[:-1], w.shape[-1] // 32, 18)
    monkeypatch.setattr(quant, "quantize_q4_0", unsigned)
    with pytest.raises(AssertionError):
        pins.test_hand_worked_block("q4_0_block.txt", "q4_0")


def test_planted_embed_off_by_one_row_is_caught(monkeypatch):
    real = om.OracleModel.embed

    def shifted(self, tokens):
        t = (np.asarray(tokens, dtype=np.int64) + 1) % self.w.vocab   # planted: next row
        return real(self, t)
    monkeypatch.setattr(om.OracleModel, "embed", shifted)
    for wtype in ("q8_0", "q4_0"):
        with pytest.raises(AssertionError):
            pins.test_embed_gathers_the_token_rows(wtype)


def _attn_block_variant(round_k_before_rope=False, round_q=False):
    """The oracle's attention block with one planted change to where the f16
    cache rounds."""
    def attn_block(self, i, h, cache, positions):
        w = self.w
        p = f"blk.{i}"
        T = h.shape[0]
        q = self.linear(h, f"{p}.attn_q").reshape(T, w.n_heads, w.head_dim).transpose(1, 0, 2)
        k = self.linear(h, f"{p}.attn_k").reshape(T, w.n_kv_heads, w.head_dim).transpose(1, 0, 2)
        v = self.linear(h, f"{p}.attn_v").reshape(T, w.n_kv_heads, w.head_dim).transpose(1, 0, 2)
        q = om.rms_norm(q, self.gain(f"{p}.attn_q_norm"), w.rms_eps)
        k = om.rms_norm(k, self.gain(f"{p}.attn_k_norm"), w.rms_eps)
        if round_k_before_rope:
            k = self.store_kv(k)
        q = om.rope(q, positions, w.rope_theta)
        k = om.rope(k, positions, w.rope_theta)
        if round_q:
            q = self.store_kv(q)
        if not round_k_before_rope:
            k = self.store_kv(k)
        v = self.store_kv(v)
        if cache[i] is not None:
            ck, cv = cache[i]
            k = np.concatenate([ck, k], axis=1)
            v = np.concatenate([cv, v], axis=1)
        cache[i] = (k, v)
        o = om.attention(q, k, v, positions)
        o = o.transpose(1, 0, 2).reshape(T, w.n_heads * w.head_dim)
        return self.linear(o, f"{p}.attn_output")
    return attn_block


def test_unplanted_variant_passes_the_store_pin(monkeypatch):
    monkeypatch.setattr(om.OracleModel, "attn_block", _attn_block_variant())
    pins.test_f16_kv_store_point_matches_torch_recomposition()


def test_planted_rounding_before_rope_is_caught(monkeypatch):
    monkeypatch.setattr(om.OracleModel, "attn_block", _attn_block_variant(round_k_before_rope=True))
    with pytest.raises(AssertionError):
        pins.test_f16_kv_store_point_matches_torch_recomposition()


def test_planted_rounding_of_q_is_caught(monkeypatch):
    monkeypatch.setattr(om.OracleModel, "attn_block", _attn_block_variant(round_q=True))
    with pytest.raises(AssertionError):
        pins.test_f16_kv_store_point_matches_torch_recomposition()


def test_planted_cutoff_without_plus_one_is_caught(monkeypatch):
    from oracle import sample as osm

    def nucleus(logits, temperature, top_p):
        z = np.asarray(logits, dtype=np.float64) / float(temperature)
        p = np.exp(z - z.max())
        p /= p.sum()
        order = np.argsort(-p, kind="stable")
        sp = p[order]
        cut = max(1, int(np.sum(np.cumsum(sp) < top_p)))   # planted: no "+ 1"
        return order[:cut], sp[:cut] / sp[:cut].sum()
    monkeypatch.setattr(osm, "nucleus", nucleus)
    with pytest.raises(AssertionError):
        pins.test_top_p_hand_worked()


def test_planted_ascending_order_is_caught(monkeypatch):
    from oracle import sample as osm

    def nucleus(logits, temperature, top_p):
        z = np.asarray(logits, dtype=np.float64) / float(temperature)
        p = np.exp(z - z.max())
        p /= p.sum()
        order = np.argsort(p, kind="stable")               # planted: ascending
        sp = p[order]
        cut = int(np.sum(np.cumsum(sp) < top_p)) + 1
        return order[:cut], sp[:cut] / sp[:cut].sum()
    monkeypatch.setattr(osm, "nucleus", nucleus)
    with pytest.raises(AssertionError):
        pins.test_top_p_hand_worked()


def test_planted_missing_temperature_is_caught(monkeypatch):
    from oracle import sample as osm
    real = osm.nucleus
    monkeypatch.setattr(osm, "nucleus", lambda l, t, p: real(l, 1.0, p))  # planted: temperature ignored
    with pytest.raises(AssertionError):
        pins.test_sampling_special_cases()


# --------------------------------------------------------------------------- sibling architectures

def test_planted_exact_gelu_is_caught(monkeypatch):
    import scipy.special
    monkeypatch.setattr(om, "gelu_tanh", lambda z: 0.5 * z * (1.0 + scipy.special.erf(z / math.sqrt(2.0))))
    with pytest.raises(AssertionError):
        pins.test_gelu_tanh_matches_torch_and_is_not_exact_gelu()
    with pytest.raises(AssertionError):
        pins.test_arch_models_match_torch_library_composition("gemma3")


def test_planted_window_off_by_one_is_caught(monkeypatch):
    real = om.attention

    def wide(q, k, v, q_pos, window=0):
        return real(q, k, v, q_pos, window + 1 if window > 0 else 0)   # planted: j >= p - window
    monkeypatch.setattr(om, "attention", wide)
    with pytest.raises(AssertionError):
        pins.test_sliding_window_attention_matches_sdpa_band_mask(3)
    with pytest.raises(AssertionError):
        pins.test_arch_models_match_torch_library_composition("gemma3")


def test_planted_inverted_layer_pattern_is_caught(monkeypatch):
    real = om.OracleModel.window_of
    monkeypatch.setattr(om.OracleModel, "window_of",
                        lambda self, i: real(self, i + 1))               # planted: global layers swapped
    with pytest.raises(AssertionError):
        pins.test_arch_models_match_torch_library_composition("gemma3")


def test_planted_missing_softcap_is_caught(monkeypatch):
    monkeypatch.setattr(om, "softcap", lambda x, c: x)
    with pytest.raises(AssertionError):
        pins.test_softcap_closed_form()
    with pytest.raises(AssertionError):
        pins.test_arch_models_match_torch_library_composition("gemma3")


def test_planted_dropped_bias_is_caught(monkeypatch):
    real = om.OracleModel.gain

    def no_bias(self, name):                                           # planted: biases dropped
        g = real(self, name)
        return g * 0.0 if name.endswith("_bias") else g
    monkeypatch.setattr(om.OracleModel, "gain", no_bias)
    with pytest.raises(AssertionError):
        pins.test_arch_models_match_torch_library_composition("qwen2")


def test_planted_qk_norm_in_llama_is_caught(monkeypatch):
    real = om.OracleModel.attn_block

    def with_norm(self, i, h, cache, positions):
        w = self.w
        object.__setattr__(w, "arch", "qwen3")                         # planted: llama with qwen3's norm
        try:
            self.weights.setdefault(f"blk.{i}.attn_q_norm", np.ones(w.head_dim, np.float32) * 1.5)
            self.weights.setdefault(f"blk.{i}.attn_k_norm", np.ones(w.head_dim, np.float32) * 1.5)
            return real(self, i, h, cache, positions)
        finally:
            object.__setattr__(w, "arch", "llama")
    monkeypatch.setattr(om.OracleModel, "attn_block", with_norm)
    with pytest.raises(AssertionError):
        pins.test_arch_models_match_torch_library_composition("llama")


# --------------------------------------------------------------------------- affine 4-bit format

def test_planted_reversed_nibble_order_is_caught(monkeypatch):
    real = quant.affine4_parts

    def reversed_parts(groups):
        q, s, b = real(groups)
        q = q.reshape(*q.shape[:-1], 8, 8)[..., ::-1].reshape(q.shape)   # planted: high nibble first
        return q, s, b
    monkeypatch.setattr(quant, "affine4_parts", reversed_parts)
    with pytest.raises(AssertionError):
        pins.test_affine4_hand_worked_group()


def test_planted_half_even_codes_are_caught(monkeypatch):
    monkeypatch.setattr(quant, "round_half_away", lambda x: np.round(x))   # numpy: halves to even
    with pytest.raises(AssertionError):
        pins.test_affine4_hand_worked_group()


def test_planted_bias_dropped_is_caught(monkeypatch):
    real = quant.bf16_value

    def deq_without_bias(blocks, wtype, dtype=np.float64):
        q, s, b = quant.affine4_parts(blocks)
        v = q.astype(dtype) * real(s).astype(dtype)[..., None]                # planted: + b missing
        return v.reshape(*blocks.shape[:-2], blocks.shape[-2] * 64)
    orig = quant.dequantize
    monkeypatch.setattr(quant, "dequantize",
                        lambda blocks, wtype, dtype=np.float64: deq_without_bias(blocks, wtype, dtype)
                        if wtype == "affine4" else orig(blocks, wtype, dtype))
    with pytest.raises(AssertionError):
        pins.test_affine4_hand_worked_group()
    with pytest.raises(AssertionError):
        pins.test_affine4_brute_force_error_bound_and_equal_groups()
