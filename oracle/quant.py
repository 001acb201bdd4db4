"""Q8_0, Q4_0 and affine 4-bit encodings, written out plainly (oracle; test infrastructure).

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

Affine 4-bit ("Alchemize PyTensor ... Gemma 3n", section on streaming the
affine-4 checkpoint): W[r, c] = q[r, c] * s[r, g(c)] + b[r, g(c)] with 4-bit q,
eight of them per uint32 word, and a bf16 scale and bias per group.  The page
gives the decoding; the readings taken for the rest:

* groups of 64 consecutive inputs of a row; element 8w + i of a group sits in
  bits 4i .. 4i + 3 of its word w (low nibble first);
* encoding in f32: s = (max - min) / 15 and b = min over the group, q =
  clamp(round((w - b) / s), 0, 15) with round-half-away and the f32 s and b;
  a group of equal values has s = 0 and q = 0; the stored s and b are bf16,
  rounded to nearest even;
* this module's record of a group is 36 bytes: the 8 words (little-endian),
  then the bf16 scale, then the bf16 bias.

Decoding q * s + b is exact in f64; in f32 the sum rounds once.
"""
from __future__ import annotations

import numpy as np

QK = 32
Q8_0_BYTES = 34
Q4_0_BYTES = 18
AFFINE_GROUP = 64
AFFINE4_BYTES = 36


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


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), rounded to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def quantize_affine4(w: np.ndarray) -> np.ndarray:
    """f32 rows [..., K] -> affine 4-bit group records [..., K/64, 36] (uint8)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert w.shape[-1] % AFFINE_GROUP == 0, "row length must be a multiple of 64"
    lead = w.shape[:-1]
    g = w.reshape(-1, AFFINE_GROUP)
    lo = np.min(g, axis=1)
    hi = np.max(g, axis=1)
    s = ((hi - lo) / np.float32(15.0)).astype(np.float32)        # f32 division
    b = lo
    safe = np.where(s == 0, np.float32(1.0), s)
    q = round_half_away(((g - b[:, None]) / safe[:, None]).astype(np.float32))
    q = np.where(s[:, None] == 0, np.float32(0.0), q)
    q = np.clip(q, 0, 15).astype(np.uint32)
    words = np.zeros((g.shape[0], 8), dtype=np.uint32)
    for i in range(8):                                            # element 8w + i at bits 4i
        words |= q[:, i::8] << np.uint32(4 * i)
    out = np.empty((g.shape[0], AFFINE4_BYTES), dtype=np.uint8)
    out[:, 0:32] = words.astype("<u4").view(np.uint8)
    out[:, 32:34] = bf16_bits(s).astype("<u2").view(np.uint8).reshape(-1, 2)
    out[:, 34:36] = bf16_bits(b).astype("<u2").view(np.uint8).reshape(-1, 2)
    return out.reshape(*lead, w.shape[-1] // AFFINE_GROUP, AFFINE4_BYTES)


def affine4_parts(groups: np.ndarray):
    """Group records [..., G, 36] -> (codes [..., G, 64] uint8, scale bf16 bits
    [..., G], bias bf16 bits [..., G])."""
    g = np.ascontiguousarray(groups)
    words = g[..., 0:32].copy().view("<u4")                      # [..., G, 8]
    q = np.empty(g.shape[:-1] + (AFFINE_GROUP,), dtype=np.uint8)
    for i in range(8):
        q[..., i::8] = (words >> np.uint32(4 * i)) & np.uint32(15)
    s = g[..., 32:34].copy().view("<u2")[..., 0]
    b = g[..., 34:36].copy().view("<u2")[..., 0]
    return q, s, b


def quantize(w: np.ndarray, wtype: str) -> np.ndarray:
    if wtype == "affine4":
        return quantize_affine4(w)
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
    """Block bytes [..., nb, 34|18] (group records [..., G, 36] for affine4)
    -> weights [..., nb*32] in ``dtype``."""
    if wtype == "affine4":
        q, s, b = affine4_parts(blocks)
        v = q.astype(dtype) * bf16_value(s).astype(dtype)[..., None] + bf16_value(b).astype(dtype)[..., None]
        return v.reshape(*blocks.shape[:-2], blocks.shape[-2] * AFFINE_GROUP)
    d = scales(blocks).astype(dtype)[..., None]
    q = codes(blocks, wtype).astype(dtype)
    if wtype == "q4_0":
        q = q - 8
    v = d * q
    return v.reshape(*blocks.shape[:-2], blocks.shape[-2] * QK)
