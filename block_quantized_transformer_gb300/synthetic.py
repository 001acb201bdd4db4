"""Seeded synthetic models built directly in device memory.

Weights come from the shared counter-based generator (``synth``: N(0, 0.02)
matrices, 1 + N(0, 0.02) gains) written on the GPU, are encoded to GGUF-order
Q8_0/Q4_0 blocks (or MLX-layout affine 4-bit groups) by the library's own
encoder (tq_quantize, tq_quantize_affine4) and repacked to the tiled layout
(tq_repack, tq_repack_affine4), in row chunks of at most 2^28 weights (a
multiple of 16 rows) so the f32 staging buffer stays at 1 GB.
"""
from __future__ import annotations

import torch

import synth

from . import QMat, Model, WTYPES, QS_BYTES, TQ_AFFINE4, quantize, quantize_affine4, tq_repack, tq_repack_affine4

CHUNK = 1 << 28


def build_matrix(w: "synth.Workload", name: str, device="cuda") -> QMat:
    wt = WTYPES[w.wtype]
    rows, cols = w.matrix_shape(name)
    nb = cols // 32
    m = QMat.empty(wt, rows, cols, device)
    step = max(16, (CHUNK // cols) // 16 * 16)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        f = torch.empty((r1 - r0) * cols, dtype=torch.float32, device=device)
        synth.dev_normal(f, w.seed, w.stream_of(name), first=r0 * cols)
        p1 = min(r0 + step, (rows + 15) // 16 * 16)  # padded rows of this chunk
        qs, d = m.qs[r0 * nb * QS_BYTES[wt]: p1 * nb * QS_BYTES[wt]], m.d[r0 * nb: p1 * nb]
        if wt == TQ_AFFINE4:
            words, scales, biases = quantize_affine4(f.view(r1 - r0, cols))
            tq_repack_affine4(words, scales, biases, r1 - r0, cols, qs, d)
            del words, scales, biases
        else:
            blocks = quantize(f.view(r1 - r0, cols), wt)
            tq_repack(wt, blocks, r1 - r0, cols, qs, d)
            del blocks
        del f
    return m


def build_gain(w: "synth.Workload", name: str, device="cuda") -> torch.Tensor:
    g = torch.empty(w.gain_len(name), dtype=torch.float32, device=device)
    synth.dev_normal(g, w.seed, w.stream_of(name), mean=1.0)
    return g


def build_bias(w: "synth.Workload", name: str, device="cuda") -> torch.Tensor:
    b = torch.empty(w.bias_len(name), dtype=torch.float32, device=device)
    synth.dev_normal(b, w.seed, w.stream_of(name), sigma=synth.BIAS_SIGMA)
    return b


def build_weights(w: "synth.Workload", device="cuda"):
    mats = {n: build_matrix(w, n, device) for n in w.matrices()}
    gains = {n: build_gain(w, n, device) for n in w.gains()}
    gains.update({n: build_bias(w, n, device) for n in w.biases()})
    return mats, gains


def build_model(w: "synth.Workload", device="cuda", max_batch=None, max_ctx=None,
                max_prefill=None, page_size=None, n_pages=None, weights=None) -> Model:
    mats, gains = weights if weights is not None else build_weights(w, device)
    return Model(vocab=w.vocab, hidden=w.hidden, n_layers=w.n_layers, n_heads=w.n_heads,
                 n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, ffn=w.ffn, wtype=w.wtype,
                 kv=w.kv, mats=mats, gains=gains,
                 max_batch=max_batch or w.batch,
                 max_ctx=max_ctx or (w.prompt_len + w.decode_steps + 1),
                 max_prefill=max_prefill or w.prompt_len,
                 page_size=(w.page_size if w.paged else 0) if page_size is None else page_size,
                 n_pages=n_pages or 0, rms_eps=w.rms_eps, rope_theta=w.rope_theta, device=device,
                 arch=w.arch, sliding_window=w.sliding_window, sliding_pattern=w.sliding_pattern,
                 logit_softcap=w.logit_softcap)
