"""GPU parity of the affine 4-bit weight format (W = q s + b per group of 64
inputs, MLX layout: "Alchemize PyTensor ... Gemma 3n"): the encoder bit-exact
against the oracle's, repack + decode exact, the GEMV and the tcgen05 GEMM
within their error bounds, and whole models of that format against the
oracle (tolerances as in test_gpu_model)."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import quant
from oracle import model as om
import block_quantized_transformer_gb300 as tq
from block_quantized_transformer_gb300.synthetic import build_model
from gpu_util import rel_logit_err, check_tokens, gpu_teacher_forced

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def special_rows(cols):
    rows = [np.zeros(cols, np.float32)]                      # equal groups: s = 0
    r = np.zeros(cols, np.float32)
    r[:5] = [-1.0, 0.875, -0.9375, 0.3, 0.0]                 # the hand-worked group (halves, clamp ends)
    rows.append(r)
    rows.append(np.full(cols, 1e-7, np.float32))             # tiny values
    rows.append(((np.arange(cols) % 64) * np.float32(0.125) - 4).astype(np.float32))  # exact codes 0..15 pattern
    return np.stack(rows)


def planar(groups):
    """Oracle group records -> (words int32 [rows][cols/8], scales, biases int16 [rows][cols/64])."""
    rows, G, _ = groups.shape
    words = np.ascontiguousarray(groups[..., 0:32]).view("<i4").reshape(rows, G * 8)
    s = np.ascontiguousarray(groups[..., 32:34]).view("<i2").reshape(rows, G)
    b = np.ascontiguousarray(groups[..., 34:36]).view("<i2").reshape(rows, G)
    return words, s, b


def qmat_of(groups, cols):
    rows = groups.shape[0]
    words, s, b = (torch.from_numpy(a.copy()).to(DEV) for a in planar(groups))
    m = tq.QMat.empty(tq.TQ_AFFINE4, rows, cols, DEV)
    tq.tq_repack_affine4(words, s, b, rows, cols, m.qs, m.d)
    return m


@pytest.mark.parametrize("rows,cols", [(257, 1024), (9, 4096)])
def test_affine4_quantize_bit_exact(rows, cols):
    w = np.concatenate([synth.host_normal(9, 78, rows * cols).reshape(rows, cols), special_rows(cols)])
    want = planar(quant.quantize_affine4(w))
    got = tq.quantize_affine4(torch.from_numpy(w).to(DEV))
    for name, a, b in zip(("words", "scales", "biases"), got, want):
        a = a.cpu().numpy()
        diff = np.argwhere(a != b)
        assert diff.size == 0, (name, diff[:10])


def test_affine4_repack_and_decode():
    rows, cols = 301, 768
    w = np.concatenate([synth.host_normal(4, 6, rows * cols).reshape(rows, cols), special_rows(cols)])
    g = quant.quantize_affine4(w)
    m = qmat_of(g, cols)
    got = tq.tq_dequantize(m).cpu().numpy()
    want = quant.dequantize(g, "affine4", np.float32)        # q s + b rounded once in f32
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.array_equal(tq.tq_dequantize(m, row0=17, n_rows=5).cpu().numpy(), want[17:22])


def _bound_check(y, x, W, r=None):
    ref = x.astype(np.float64) @ W.T
    bound = np.abs(x.astype(np.float64)) @ np.abs(W).T
    tol = (2.0 ** -10 + x.shape[1] * 2.0 ** -23) * bound + 2.0 ** -25 * np.abs(x).sum(1, keepdims=True)
    if r is not None:
        ref = ref + r
        tol = tol + 2.0 ** -23 * np.abs(r)
    err = np.abs(y - ref)
    assert np.all(err <= tol), float(np.max(err / tol))


@pytest.mark.parametrize("rows,cols,n", [(4096 + 5, 4096, 1), (77, 3072, 3), (1003, 12288, 1), (33, 256, 2)])
def test_affine4_gemv_matches_oracle(rows, cols, n):
    w = synth.host_normal(rows, 1, rows * cols).reshape(rows, cols)
    g = quant.quantize_affine4(w)
    m = qmat_of(g, cols)
    x = synth.host_normal(rows, 2, n * cols, sigma=1.0).reshape(n, cols)
    r = synth.host_normal(rows, 3, n * rows, sigma=1.0).reshape(n, rows) if n > 1 else None
    y = tq.tq_gemv(m, torch.from_numpy(x).to(DEV),
                   residual=None if r is None else torch.from_numpy(r).to(DEV)).cpu().numpy()
    _bound_check(y, x, quant.dequantize(g, "affine4"), r)


@pytest.mark.parametrize("rows,cols,n", [(4096 + 5, 4096, 37), (1003, 12288, 5), (6144, 4096, 2048),
                                         (256, 12288, 32), (130, 256, 2)])
def test_affine4_gemm_matches_oracle(rows, cols, n):
    w = synth.host_normal(rows + n, 1, rows * cols).reshape(rows, cols)
    g = quant.quantize_affine4(w)
    m = qmat_of(g, cols)
    x = synth.host_normal(rows + n, 2, n * cols, sigma=1.0).reshape(n, cols)
    x[0, :] *= 1e-3
    y = tq.tq_gemm(m, torch.from_numpy(x).to(DEV)).cpu().numpy()
    _bound_check(y, x, quant.dequantize(g, "affine4"))


@pytest.mark.parametrize("kv,prompt_len,steps", [("f32", 8, 16), ("f16", 120, 8)])
def test_affine4_model_matches_oracle(kv, prompt_len, steps):
    w = dataclasses.replace(synth.TINY, name=f"tiny_affine4_{kv}", wtype="affine4", kv=kv)
    prompt = list(w.prompt(n=prompt_len))
    ref = om.OracleModel(w, om.synth_weights(w))
    toks, ref_logits = om.run_greedy(ref, prompt, steps)
    model = build_model(w, device=DEV, max_ctx=prompt_len + steps + 1, max_prefill=prompt_len)
    got_l, got_t = gpu_teacher_forced(model, prompt, toks[:steps], DEV)
    assert model.status() == 0
    model.close()
    tol = 2e-3 if kv == "f32" else 1e-2
    errs = [rel_logit_err(a, b) for a, b in zip(got_l, ref_logits)]
    print(f"affine4 {kv}: max rel logit err {max(errs):.2e}")
    assert max(errs) <= tol, (max(errs), int(np.argmax(errs)))
    check_tokens(got_t, ref_logits, tol)


def test_affine4_device_weights_match_oracle_encoding():
    # the model's matrices (device generator + the library's encoder + repack)
    # decode to exactly the oracle's own encoding of the host generator's weights
    w = dataclasses.replace(synth.TINY, name="tiny_affine4", wtype="affine4")
    from block_quantized_transformer_gb300.synthetic import build_matrix
    for name in ("token_embd", "blk.1.ffn_down", "blk.0.attn_q"):
        m = build_matrix(w, name, DEV)
        got = tq.tq_dequantize(m).cpu().numpy()
        want = quant.dequantize(quant.quantize_affine4(synth.host_tensor(w, name)), "affine4", np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), name
