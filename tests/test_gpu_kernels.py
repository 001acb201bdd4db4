"""GPU parity of the single kernels against the oracle, through the C ABI:
encoding and decoding bit-exact; GEMV and LM head within f32 error bounds;
argmax ties to the lowest index."""
import numpy as np
import pytest
import torch

import synth
from oracle import quant
import block_quantized_transformer_gb300 as tq
from block_quantized_transformer_gb300.synthetic import build_matrix

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
WT = {"q8_0": tq.TQ_Q8_0, "q4_0": tq.TQ_Q4_0}


def special_rows(cols):
    """Rows exercising ties, halves, zeros and signed extremes."""
    rows = []
    z = np.zeros(cols, np.float32)
    rows.append(z.copy())                                  # all-zero blocks
    r = np.zeros(cols, np.float32)
    r[0], r[1] = 0.0625, -0.0625                           # Q4_0 extreme tie: first wins
    rows.append(r)
    r = np.zeros(cols, np.float32)
    r[3], r[10] = -0.0625, 0.0625
    rows.append(r)
    u = np.float32(2.0 ** -10)
    r = (np.arange(cols) % 32 - 15.5).astype(np.float32) * u   # x.5 multiples of the step
    r[::32] = 127 * u
    rows.append(r)
    r = (np.arange(cols) % 16 - 7.5).astype(np.float32) * np.float32(2.0 ** -7)
    r[::32] = -8 * np.float32(2.0 ** -7)
    rows.append(r)
    r = np.full(cols, 1e-7, np.float32)                    # tiny: subnormal fp16 scales
    rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", [(257, 1024), (9, 4096)])
def test_quantize_bit_exact(wtype, rows, cols):
    w = synth.host_normal(9, 77, rows * cols).reshape(rows, cols)
    w = np.concatenate([w, special_rows(cols)])
    want = quant.quantize(w, wtype)
    got = tq.quantize(torch.from_numpy(w).to(DEV), WT[wtype]).cpu().numpy()
    assert got.shape == want.shape
    diff = np.argwhere(got != want)
    assert diff.size == 0, diff[:10]


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_repack_and_decode_bit_exact(wtype):
    rows, cols = 301, 768
    w = np.concatenate([synth.host_normal(4, 5, rows * cols).reshape(rows, cols), special_rows(cols)])
    blocks = quant.quantize(w, wtype)
    m = tq.QMat.from_blocks(WT[wtype], torch.from_numpy(blocks).to(DEV), w.shape[0], cols)
    got = tq.tq_dequantize(m).cpu().numpy()
    want = quant.dequantize(blocks, wtype, np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    part = tq.tq_dequantize(m, row0=17, n_rows=5).cpu().numpy()
    assert np.array_equal(part, want[17:22])


def _gemv_case(wtype, rows, cols, batch, residual, seed):
    w = synth.host_normal(seed, 1, rows * cols).reshape(rows, cols)
    blocks = quant.quantize(w, wtype)
    m = tq.QMat.from_blocks(WT[wtype], torch.from_numpy(blocks).to(DEV), rows, cols)
    x = synth.host_normal(seed, 2, batch * cols, sigma=1.0).reshape(batch, cols)
    r = synth.host_normal(seed, 3, batch * rows, sigma=1.0).reshape(batch, rows) if residual else None
    y = tq.tq_gemv(m, torch.from_numpy(x).to(DEV),
                   residual=None if r is None else torch.from_numpy(r).to(DEV)).cpu().numpy()
    W = quant.dequantize(blocks, wtype)
    ref = x.astype(np.float64) @ W.T
    bound = np.abs(x.astype(np.float64)) @ np.abs(W).T
    # fp16 operands: weight and activation each rounded once to 11 significant
    # bits (2^-10 of |x w| together), weights below 2^-14 rounded to a multiple
    # of 2^-24, and an allowance of 2^-23 per input for the f32 sums
    tol = (2.0 ** -10 + cols * 2.0 ** -23) * bound + 2.0 ** -25 * np.abs(x).sum(1, keepdims=True)
    if r is not None:
        ref = ref + r
        tol = tol + 2.0 ** -23 * np.abs(r)
    err = np.abs(y - ref)
    assert np.all(err <= tol), float(np.max(err / tol))
    return float(np.max(err / np.maximum(bound, 1e-30)))


@pytest.mark.parametrize("wtype,rows,cols", [
    ("q4_0", 4096 + 5, 4096), ("q4_0", 1003, 12288), ("q4_0", 129, 1024), ("q4_0", 77, 3072),
    ("q8_0", 300, 1024), ("q8_0", 77, 3072), ("q8_0", 130, 256), ("q8_0", 50, 768),
    ("q8_0", 64, 2048), ("q4_0", 33, 256), ("q8_0", 1, 4096)])
def test_gemv_matches_oracle(wtype, rows, cols):
    _gemv_case(wtype, rows, cols, 1, False, rows + cols)


@pytest.mark.parametrize("batch", [2, 5])
def test_gemv_batched_with_residual(batch):
    _gemv_case("q4_0", 515, 2048, batch, True, 11)
    _gemv_case("q8_0", 200, 1024, batch, True, 12)


def _gemm_case(wtype, rows, cols, n, residual, seed):
    w = synth.host_normal(seed, 1, rows * cols).reshape(rows, cols)
    blocks = quant.quantize(w, wtype)
    m = tq.QMat.from_blocks(WT[wtype], torch.from_numpy(blocks).to(DEV), rows, cols)
    x = synth.host_normal(seed, 2, n * cols, sigma=1.0).reshape(n, cols)
    x[0, :] *= 1e-3                                   # rows of very different scales
    r = synth.host_normal(seed, 3, n * rows, sigma=1.0).reshape(n, rows) if residual else None
    y = tq.tq_gemm(m, torch.from_numpy(x).to(DEV),
                   residual=None if r is None else torch.from_numpy(r).to(DEV)).cpu().numpy()
    W = quant.dequantize(blocks, wtype)
    ref = x.astype(np.float64) @ W.T
    bound = np.abs(x.astype(np.float64)) @ np.abs(W).T
    # fp16 operands: weight and activation each rounded once to 11 significant
    # bits (2^-10 of |x w| together), weights below 2^-14 rounded to a multiple
    # of 2^-24, and an allowance of 2^-23 per input for the f32 sums
    tol = (2.0 ** -10 + cols * 2.0 ** -23) * bound + 2.0 ** -25 * np.abs(x).sum(1, keepdims=True)
    if r is not None:
        ref = ref + r
        tol = tol + 2.0 ** -23 * np.abs(r)
    err = np.abs(y - ref)
    assert np.all(err <= tol), float(np.max(err / tol))
    return float(np.max(err / np.maximum(bound, 1e-30)))


@pytest.mark.parametrize("wtype,rows,cols,n", [
    ("q4_0", 4096 + 5, 4096, 37), ("q4_0", 77, 3072, 33), ("q4_0", 1003, 12288, 5),
    ("q4_0", 130, 256, 2), ("q8_0", 300, 1024, 64), ("q8_0", 50, 768, 31), ("q8_0", 1, 4096, 3),
    ("q4_0", 1024 + 16, 4096, 300), ("q8_0", 384, 1024, 257), ("q4_0", 6144, 4096, 2048),
    ("q4_0", 256, 12288, 96), ("q8_0", 200, 512, 128)])
def test_gemm_matches_oracle(wtype, rows, cols, n):
    _gemm_case(wtype, rows, cols, n, False, rows + cols + n)


def test_gemm_with_residual():
    _gemm_case("q4_0", 515, 2048, 70, True, 13)
    _gemm_case("q8_0", 200, 1024, 9, True, 14)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_lm_head_logits_and_argmax_ties(wtype):
    vocab, hidden = 20011, 1024
    w = synth.host_normal(21, 1, vocab * hidden).reshape(vocab, hidden)
    blocks = quant.quantize(w, wtype)
    x = synth.host_normal(21, 2, 2 * hidden, sigma=1.0).reshape(2, hidden)
    g = synth.host_normal(21, 3, hidden, mean=1.0)
    W = quant.dequantize(blocks, wtype)
    xn = x.astype(np.float64) / np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True) + 1e-6) * g
    ref = xn @ W.T
    top = int(np.argmax(ref[0]))
    # plant an exact tie for row 0: copy the winning row to a lower index
    low = max(0, top - 1 - (top // 2))
    blocks[low] = blocks[top]
    ref = xn @ quant.dequantize(blocks, wtype).T
    m = tq.QMat.from_blocks(WT[wtype], torch.from_numpy(blocks).to(DEV), vocab, hidden)
    logits, am = tq.tq_lm_head(m, torch.from_numpy(x).to(DEV), torch.from_numpy(g).to(DEV))
    lg = logits.double().cpu().numpy()
    for b in range(2):
        assert np.max(np.abs(lg[b] - ref[b])) <= 1e-5 * (ref[b].max() - ref[b].min())
        assert int(am[b]) == int(np.argmax(lg[b]))          # exact argmax of its own logits
    assert int(am[0]) == low                                 # tie -> lowest index
    _, am2 = tq.tq_lm_head(m, torch.from_numpy(x).to(DEV), torch.from_numpy(g).to(DEV),
                           want_logits=False)
    assert torch.equal(am, am2)


@pytest.mark.parametrize("wl", synth.WORKLOADS[:4], ids=lambda w: w.name)
def test_device_generator_and_encoder_match_host(wl):
    """The GPU model's inputs equal the oracle's: device generator == host
    generator, and the GPU encoder == the oracle's encoder, on sampled rows of
    every tensor kind of each workload."""
    for name in ["token_embd", "blk.0.attn_q", f"blk.{wl.n_layers - 1}.ffn_down"]:
        rows, cols = wl.matrix_shape(name)
        for r0 in (0, rows - 3):
            host = synth.host_tensor(wl, name, rows=slice(r0, r0 + 3))
            dev = torch.empty(3 * cols, dtype=torch.float32, device=DEV)
            synth.dev_normal(dev, wl.seed, wl.stream_of(name), first=r0 * cols)
            d = dev.cpu().numpy().reshape(3, cols)
            assert np.array_equal(d.view(np.uint32), host.view(np.uint32))
            got = tq.quantize(dev.view(3, cols), WT[wl.wtype]).cpu().numpy()
            assert np.array_equal(got, quant.quantize(host, wl.wtype))
    g = torch.empty(wl.hidden, dtype=torch.float32, device=DEV)
    synth.dev_normal(g, wl.seed, wl.stream_of("output_norm"), mean=1.0)
    assert np.array_equal(g.cpu().numpy(), synth.host_tensor(wl, "output_norm"))
    m = build_matrix(wl, "blk.0.attn_k", DEV)
    want = quant.dequantize(quant.quantize(synth.host_tensor(wl, "blk.0.attn_k"), wl.wtype),
                            wl.wtype, np.float32)
    assert np.array_equal(tq.tq_dequantize(m).cpu().numpy(), want)
