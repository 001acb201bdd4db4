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
