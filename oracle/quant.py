"""Q8_0 and Q4_0 block encodings, written out plainly (oracle; test infrastructure).

The pages name GGUF weights and say that large weights stay quantized and are
multiplied in f32 after decoding ("Inferencia local y arquitecturas", section
"Elegir el motor"; "PyTensor Más Allá de PyMC", GGUF loading), but they print
neither block format.  The workload descriptions define both:

* Q8_0: blocks of 32 weights along the input dimension; one fp16 scale
  d = max|w| / 127 and int8 q = round(w / d); value d * q.
* Q4_0: blocks of 32; fp16 scale d = m / -8 with m the weight of largest
  magnitude taken with its sign; 4-bit q = clamp(round(w / d) + 8, 0, 15);
  value d * (q - 8).

Readings where the definition is open:

* d is computed in f32, w / d is an f32 division by that f32 d, and the
  stored scale is fp16(d) rounded to nearest even.
* round() is round-half-away-from-zero (C ``round``).
* Q8_0 codes are clamped to [-127, 127]; Q4_0 codes to [0, 15].
* Q4_0's extreme m is the first element of largest |w| in index order.
* an all-zero block has d = 0 and q = 0 (Q8_0) or 8 (Q4_0).
* byte layout (GGUF-style, little-endian): Q8_0 = fp16 d, int8 q[32] (34 B);
  Q4_0 = fp16 d, uint8 qs[16] with qs[j] = q[j] | q[j+16] << 4 (18 B).

Decoding is exact in f32 and f64: an fp16 significand (11 bits) times an
integer of at most 8 bits.
"""
from __future__ import annotations

import numpy as np

QK = 32
Q8_0_BYTES = 34
Q4_0_BYTES = 18


def round_half_away(x: np.ndarray) -> np.ndarray:
    """Round to the nearest integer, halves away from zero, in x's precision."""
    t = np.trunc(x)
    frac = x - t                      # exact for |x| < 2**23 in f32
    return t + np.where(np.abs(frac) >= 0.5, np.sign(x), 0).astype(x.dtype)


def _blocks(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert w.shape[-1] % QK == 0, "row length must be a multiple of 32"
    return w.reshape(-1, QK)


def quantize_q8_0(w: np.ndarray) -> np.ndarray:
    """f32 rows [..., K] -> Q8_0 block bytes [..., K/32, 34] (uint8)."""
    lead = w.shape[:-1]
    b = _blocks(w)
    amax = np.max(np.abs(b), axis=1)                          # f32
    d = (amax / np.float32(127.0)).astype(np.float32)          # f32 division
    safe = np.where(d == 0, np.float32(1.0), d)
    q = round_half_away((b / safe[:, None]).astype(np.float32))
    q = np.where(d[:, None] == 0, np.float32(0.0), q)
    q = np.clip(q, -127, 127).astype(np.int8)
    out = np.empty((b.shape[0], Q8_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(-1, 2)
    out[:, 2:] = q.view(np.uint8)
    return out.reshape(*lead, w.shape[-1] // QK, Q8_0_BYTES)


def quantize_q4_0(w: np.ndarray) -> np.ndarray:
    """f32 rows [..., K] -> Q4_0 block bytes [..., K/32, 18] (uint8)."""
    lead = w.shape[:-1]
    b = _blocks(w)
    idx = np.argmax(np.abs(b), axis=1)                         # first of the largest
    m = b[np.arange(b.shape[0]), idx]
    d = (m / np.float32(-8.0)).astype(np.float32)
    safe = np.where(d == 0, np.float32(1.0), d)
    q = round_half_away((b / safe[:, None]).astype(np.float32)) + np.float32(8.0)
    q = np.where(d[:, None] == 0, np.float32(8.0), q)
    q = np.clip(q, 0, 15).astype(np.uint8)
    out = np.empty((b.shape[0], Q4_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(-1, 2)
    out[:, 2:] = q[:, :16] | (q[:, 16:] << 4)
    return out.reshape(*lead, w.shape[-1] // QK, Q4_0_BYTES)


def quantize(w: np.ndarray, wtype: str) -> np.ndarray:
    return quantize_q8_0(w) if wtype == "q8_0" else quantize_q4_0(w)


def scales(blocks: np.ndarray) -> np.ndarray:
    """The fp16 scale of every block, as float16."""
    return np.ascontiguousarray(blocks[..., 0:2]).view(np.float16)[..., 0]


def codes(blocks: np.ndarray, wtype: str) -> np.ndarray:
    """Integer codes [..., K/32, 32]: int8 q (Q8_0) or uint8 q in 0..15 (Q4_0)."""
    if wtype == "q8_0":
        return np.ascontiguousarray(blocks[..., 2:]).view(np.int8)
    qs = blocks[..., 2:]
    return np.concatenate([qs & 0x0F, qs >> 4], axis=-1)


def dequantize(blocks: np.ndarray, wtype: str, dtype=np.float64) -> np.ndarray:
    """Block bytes [..., nb, 34|18] -> weights [..., nb*32] in ``dtype``."""
    d = scales(blocks).astype(dtype)[..., None]
    q = codes(blocks, wtype).astype(dtype)
    if wtype == "q4_0":
        q = q - 8
    v = d * q
    return v.reshape(*blocks.shape[:-2], blocks.shape[-2] * QK)
