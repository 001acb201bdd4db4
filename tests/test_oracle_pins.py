"""Pins of the oracle to facts that do not come from the oracle itself:
hand-worked blocks, closed forms, invariants, library routines and brute force.
Each test is chosen so that a plausible slip (a dropped term, a wrong sign,
index, rounding mode or operand order) fails it."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from conftest import golden
from oracle import quant
from oracle import model as om


# --------------------------------------------------------------------------- quant

def _fixture(name):
    g = golden(name)
    unit = float(g["unit"][0][0])
    w = (np.array([float(v) for v in g["w"][0]], dtype=np.float64) * unit).astype(np.float32)
    raw = bytes(int(b, 16) for b in g["bytes"][0])
    values = np.array([float(v) for v in g["values"][0]]) * unit
    return w, raw, values


@pytest.mark.parametrize("name,wtype", [("q8_0_block.txt", "q8_0"), ("q4_0_block.txt", "q4_0")])
def test_hand_worked_block(name, wtype):
    w, raw, values = _fixture(name)
    blk = quant.quantize(w[None, :], wtype)
    assert blk.shape == (1, 1, 34 if wtype == "q8_0" else 18)
    assert bytes(blk.reshape(-1)) == raw
    deq = quant.dequantize(np.frombuffer(raw, np.uint8).reshape(1, 1, -1), wtype)
    assert np.array_equal(deq.reshape(-1), values)


def test_round_half_away():
    x = np.array([0.5, 1.5, 2.5, -0.5, -2.5, 0.49999997, -0.49999997, 126.5, -127.0],
                 dtype=np.float32)
    assert quant.round_half_away(x).tolist() == [1, 2, 3, -1, -3, 0, 0, 127, -127]


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_zero_block(wtype):
    blk = quant.quantize(np.zeros((1, 32), np.float32), wtype)
    assert quant.scales(blk).item() == 0.0
    assert np.all(quant.dequantize(blk, wtype) == 0.0)
    q = quant.codes(blk, wtype)
    assert np.all(q == (0 if wtype == "q8_0" else 8))


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_brute_force_codes_and_error_bound(wtype):
    """Codes recomputed element by element in f64 straight from the definition
    agree with the encoder (except where w/d sits within 1e-5 of a rounding
    boundary, where f32 and f64 may decide differently); every unclamped
    decoded weight lies within half a step of the original, up to the fp16
    rounding of the scale."""
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((512, 64)) * 0.02).astype(np.float32)
    w[3, :32] *= 1e-3                      # a block of tiny values (small fp16 scale)
    blk = quant.quantize(w, wtype)
    d16 = quant.scales(blk).astype(np.float64).reshape(512, 2)
    q = quant.codes(blk, wtype).astype(np.int64).reshape(512, 2, 32)
    wb = w.astype(np.float64).reshape(512, 2, 32)
    n_checked = 0
    for r in range(512):
        for b in range(2):
            x = wb[r, b]
            if wtype == "q8_0":
                d = np.abs(x).max() / 127.0
                lo, hi, off = -127, 127, 0
            else:
                i = int(np.argmax(np.abs(x)))
                d = x[i] / -8.0
                lo, hi, off = 0, 15, 8
            for j in range(32):
                t = x[j] / d
                frac = abs(t) - math.floor(abs(t))
                if abs(frac - 0.5) < 1e-5:
                    continue
                want = min(hi, max(lo, int(math.copysign(math.floor(abs(t) + 0.5), t)) + off))
                assert q[r, b, j] == want, (r, b, j)
                n_checked += 1
                qq = want - off
                if lo < want < hi or wtype == "q8_0":
                    assert abs(x[j] - d16[r, b] * qq) <= abs(d) / 2 * (1 + 1e-5) + \
                        abs(qq) * abs(abs(d16[r, b]) - abs(d)) + 1e-15
    assert n_checked > 0.99 * 512 * 64
    if wtype == "q8_0":
        assert np.all(np.abs(q).max(axis=-1) == 127)
    else:
        idx = np.argmax(np.abs(wb), axis=-1)
        assert np.all(np.take_along_axis(q, idx[..., None], axis=-1) == 0)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_dequant_exact_in_f32(wtype):
    """fp16 scale x small integer is exact in f32: f32 and f64 decodes agree bit for bit."""
    w = synth.host_normal(3, 3, 4096 * 4).reshape(4, 4096)
    blk = quant.quantize(w, wtype)
    assert np.array_equal(quant.dequantize(blk, wtype, np.float32).astype(np.float64),
                          quant.dequantize(blk, wtype, np.float64))


# --------------------------------------------------------------------------- rmsnorm

def test_rms_norm_closed_form():
    c, eps, H = 0.37, 1e-6, 64
    g = np.linspace(0.5, 1.5, H)
    y = om.rms_norm(np.full(H, c), g, eps)
    assert np.allclose(y, c / math.sqrt(c * c + eps) * g, rtol=1e-15, atol=0)


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 256))
    g = 1 + 0.02 * rng.standard_normal(256)
    ref = F.rms_norm(torch.from_numpy(x), (256,), weight=torch.from_numpy(g), eps=1e-6).numpy()
    assert np.allclose(om.rms_norm(x, g, 1e-6), ref, rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------- rope

def test_rope_closed_form_pairs_and_frequencies():
    """hd=4, theta=1e6: pairs are (0,2) and (1,3) with frequencies 1 and 1e-3."""
    e0 = np.array([[1.0, 0, 0, 0]])
    e1 = np.array([[0, 1.0, 0, 0]])
    e2 = np.array([[0, 0, 1.0, 0]])
    assert np.allclose(om.rope(e0, [1], 1e6), [[math.cos(1), 0, math.sin(1), 0]], atol=1e-15)
    assert np.allclose(om.rope(e2, [1], 1e6), [[-math.sin(1), 0, math.cos(1), 0]], atol=1e-15)
    assert np.allclose(om.rope(e1, [1000], 1e6), [[0, math.cos(1), 0, math.sin(1)]], atol=1e-12)


def test_rope_equals_complex_rotation():
    """Half-split RoPE = multiplying (x_i + i x_{i+hd/2}) by exp(i * pos * theta^(-i/(hd/2)))."""
    rng = np.random.default_rng(1)
    hd, T = 128, 9
    x = rng.standard_normal((3, T, hd))
    pos = np.array([0, 1, 2, 7, 100, 1000, 4095, 8191, 262143])
    z = x[..., : hd // 2] + 1j * x[..., hd // 2:]
    f = 1e6 ** (-np.arange(hd // 2) / (hd // 2))
    zr = z * np.exp(1j * pos[:, None] * f[None, :])
    ref = np.concatenate([zr.real, zr.imag], axis=-1)
    # angles up to 2.6e5 rad: one ulp of the frequency moves them by ~1e-10
    assert np.allclose(om.rope(x, pos, 1e6), ref, rtol=0, atol=1e-9)


def test_rope_invariants():
    rng = np.random.default_rng(2)
    hd = 64
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))
    assert np.allclose(om.rope(q, [0], 1e6), q, atol=0)                    # p = 0 identity
    for p in [1, 17, 4000]:
        assert np.isclose(np.linalg.norm(om.rope(q, [p], 1e6)), np.linalg.norm(q), rtol=1e-13)
    m, n, s = 37, 5, 911
    a = np.sum(om.rope(q, [m], 1e6) * om.rope(k, [n], 1e6))
    b = np.sum(om.rope(q, [m + s], 1e6) * om.rope(k, [n + s], 1e6))
    assert np.isclose(a, b, rtol=1e-11)


# --------------------------------------------------------------------------- attention

def _sdpa(q, k, v, causal):
    G = q.shape[0] // k.shape[0]
    kk = torch.from_numpy(k).repeat_interleave(G, dim=0)
    vv = torch.from_numpy(v).repeat_interleave(G, dim=0)
    return F.scaled_dot_product_attention(torch.from_numpy(q), kk, vv, is_causal=causal).numpy()


@pytest.mark.parametrize("nq,nkv", [(4, 2), (8, 2), (16, 8), (4, 4), (4, 1)])
def test_attention_prefill_matches_sdpa(nq, nkv):
    rng = np.random.default_rng(nq * 10 + nkv)
    T, hd = 13, 32
    q, k, v = (rng.standard_normal((n, T, hd)) for n in (nq, nkv, nkv))
    out = om.attention(q, k, v, np.arange(T))
    assert np.allclose(out, _sdpa(q, k, v, True), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("nq,nkv", [(32, 8), (16, 8), (4, 2)])
def test_attention_decode_matches_sdpa(nq, nkv):
    rng = np.random.default_rng(7)
    S, hd = 300, 128
    q = rng.standard_normal((nq, 1, hd))
    k, v = (rng.standard_normal((nkv, S, hd)) for _ in range(2))
    out = om.attention(q, k, v, np.array([S - 1]))
    assert np.allclose(out, _sdpa(q, k, v, False), rtol=1e-12, atol=1e-13)


def test_gqa_group_one_is_mha_and_rows_sum_to_one():
    rng = np.random.default_rng(3)
    T, hd, n = 6, 16, 4
    q, k, v = (rng.standard_normal((n, T, hd)) for _ in range(3))
    ref = np.stack([om.softmax(np.where(np.tril(np.ones((T, T))) > 0,
                                        q[h] @ k[h].T / math.sqrt(hd), -np.inf)) @ v[h]
                    for h in range(n)])
    assert np.allclose(om.attention(q, k, v, np.arange(T)), ref, rtol=1e-13)
    p = om.softmax(rng.standard_normal((5, 77)) * 30)
    assert np.allclose(p.sum(-1), 1.0, rtol=0, atol=1e-15)


def test_silu_matches_torch():
    z = np.linspace(-30, 30, 1001)
    assert np.allclose(om.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)


def test_argmax_lowest_index_on_ties():
    assert om.argmax(np.array([1.0, 3.0, 3.0, -1.0])) == 1
    x = np.zeros(151936)
    x[[5, 77, 150000]] = 2.0
    assert om.argmax(x) == 5


# --------------------------------------------------------------------------- whole model

def _tiny(kv="f32", seed=0, n_heads=4, n_kv=2):
    w = synth.Workload("pin", vocab=512, hidden=128, n_layers=2, n_heads=n_heads,
                       n_kv_heads=n_kv, head_dim=32, ffn=256, wtype="q8_0", kv=kv, seed=seed)
    return w, om.OracleModel(w, om.synth_weights(w))


@pytest.mark.parametrize("kv", ["f32", "f16"])
def test_cached_decode_equals_full_recompute(kv):
    """KV-cached decode = rebuilding the whole prefix with no state, every step."""
    w, m = _tiny(kv)
    prompt = list(w.prompt(n=5))
    toks, logits = om.run_greedy(m, prompt, 6)
    seq = prompt + toks[:-1]
    for s in range(7):
        ref = m.forward_nocache(seq[: len(prompt) + s])
        assert np.allclose(logits[s], ref, rtol=1e-12, atol=1e-12), s


def test_prefill_split_equals_one_shot():
    """Prefilling in two chunks gives the same cache and logits as one call."""
    w, m = _tiny()
    prompt = list(w.prompt(n=9))
    c1 = m.new_cache()
    a = m.forward(prompt, c1, 0)
    c2 = m.new_cache()
    m.forward(prompt[:4], c2, 0)
    b = m.forward(prompt[4:], c2, 4)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)
    for (k1, v1), (k2, v2) in zip(c1, c2):
        assert np.allclose(k1, k2, atol=1e-14) and np.allclose(v1, v2, atol=1e-14)


def test_model_matches_torch_library_composition():
    """Whole forward recomposed from torch library routines (F.rms_norm, SDPA with
    repeat_interleave, F.silu, torch.matmul) on the oracle's decoded weights."""
    w, m = _tiny(n_heads=4, n_kv=2)
    prompt = list(w.prompt(n=7))
    T, hd = len(prompt), w.head_dim

    def W(n):
        return torch.from_numpy(m.matrix(n))

    def g(n):
        return torch.from_numpy(m.gain(n))

    x = torch.from_numpy(m.embed(prompt))
    pos = np.arange(T)
    ang = torch.from_numpy(om.rope_angles(pos, hd, w.rope_theta))
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rot(t):
        a, b = t[..., : hd // 2], t[..., hd // 2:]
        return torch.cat([a * cos - b * sin, a * sin + b * cos], -1)

    for i in range(w.n_layers):
        p = f"blk.{i}"
        h = F.rms_norm(x, (w.hidden,), weight=g(f"{p}.attn_norm"), eps=w.rms_eps)
        q = (h @ W(f"{p}.attn_q").T).view(T, w.n_heads, hd).transpose(0, 1)
        k = (h @ W(f"{p}.attn_k").T).view(T, w.n_kv_heads, hd).transpose(0, 1)
        v = (h @ W(f"{p}.attn_v").T).view(T, w.n_kv_heads, hd).transpose(0, 1)
        q = rot(F.rms_norm(q, (hd,), weight=g(f"{p}.attn_q_norm"), eps=w.rms_eps))
        k = rot(F.rms_norm(k, (hd,), weight=g(f"{p}.attn_k_norm"), eps=w.rms_eps))
        o = F.scaled_dot_product_attention(q, k.repeat_interleave(w.group, 0),
                                           v.repeat_interleave(w.group, 0), is_causal=True)
        x = x + o.transpose(0, 1).reshape(T, -1) @ W(f"{p}.attn_output").T
        h = F.rms_norm(x, (w.hidden,), weight=g(f"{p}.ffn_norm"), eps=w.rms_eps)
        x = x + (F.silu(h @ W(f"{p}.ffn_gate").T) * (h @ W(f"{p}.ffn_up").T)) @ W(f"{p}.ffn_down").T
    xl = F.rms_norm(x[-1], (w.hidden,), weight=g("output_norm"), eps=w.rms_eps)
    ref = (xl @ W("token_embd").T).numpy()
    assert np.allclose(m.forward_nocache(prompt), ref, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------- embedding, KV store

def _decode_row_by_hand(raw_row: np.ndarray, wtype: str) -> list:
    """One row of GGUF-order blocks decoded byte by byte in plain Python,
    independently of oracle.quant: fp16 scale, then int8 codes (Q8_0) or
    nibble pairs, low nibble = element j, high nibble = element j + 16 (Q4_0)."""
    import struct
    out = []
    for blk in raw_row:
        b = bytes(int(v) for v in blk)
        d = struct.unpack("<e", b[:2])[0]
        if wtype == "q8_0":
            out += [d * struct.unpack("<b", b[2 + j:3 + j])[0] for j in range(32)]
        else:
            lo = [(b[2 + j] & 15) - 8 for j in range(16)]
            hi = [(b[2 + j] >> 4) - 8 for j in range(16)]
            out += [d * q for q in lo + hi]
    return out


@pytest.mark.parametrize("wtype", ["q8_0", "q4_0"])
def test_embed_gathers_the_token_rows(wtype):
    """embed(t) is row t of token_embd, decoded: checked against a byte-by-byte
    decode of that row and against the generator's f32 row t (within one
    quantization step: half a step of rounding, the fp16 rounding of the scale,
    and Q4_0's clamp of +8 steps to +7), which rows t - 1 and t + 1 are not."""
    w = synth.Workload("pin_embed", vocab=300, hidden=64, n_layers=1, n_heads=2, n_kv_heads=1,
                       head_dim=32, ffn=64, wtype=wtype, kv="f32", seed=4)
    m = om.OracleModel(w, om.synth_weights(w))
    tokens = [0, 1, 299, 150, 150, 7]
    x = m.embed(tokens)
    assert x.shape == (len(tokens), w.hidden)
    f32 = synth.host_tensor(w, "token_embd").astype(np.float64)
    raw = m.weights["token_embd"]
    for i, t in enumerate(tokens):
        assert x[i].tolist() == _decode_row_by_hand(raw[t], wtype), (i, t)
        err = np.abs(x[i] - f32[t]).reshape(-1, 32).max(axis=1)
        step = np.abs(f32[t]).reshape(-1, 32).max(axis=1) / (127.0 if wtype == "q8_0" else 8.0)
        assert np.all(err <= 1.01 * step), (t, err / step)
        for nb in (t - 1, t + 1):
            if 0 <= nb < w.vocab:
                assert np.abs(x[i] - f32[nb]).max() > 4 * step.max()


def test_f16_kv_store_point_matches_torch_recomposition():
    """With an f16 cache, K is rounded to f16 after QK-RMSNorm and RoPE, V after
    its projection, and q is not rounded.  Recomposed with torch (f64
    F.rms_norm, rotation as a complex multiply, Tensor.half) from the oracle's
    decoded weights: the cache holds exactly the recomposed K/V, and the
    layer's attention output equals SDPA over unrounded q and rounded K/V."""
    w, m = _tiny("f16")
    prompt = list(w.prompt(n=6))
    T, hd, half = len(prompt), w.head_dim, w.head_dim // 2
    x = m.embed(prompt)
    p = "blk.0"
    h = om.rms_norm(x, m.gain(f"{p}.attn_norm"), w.rms_eps)
    cache = m.new_cache()
    out = m.attn_block(0, h, cache, np.arange(T))

    def W(n):
        return torch.from_numpy(m.matrix(n))

    th = torch.from_numpy(h)
    ang = torch.from_numpy(om.rope_angles(np.arange(T), hd, w.rope_theta))
    turn = torch.polar(torch.ones_like(ang), ang)                      # e^{i angle}

    def rot(t):
        z = torch.complex(t[..., :half], t[..., half:]) * turn
        return torch.cat([z.real, z.imag], -1)

    q = (th @ W(f"{p}.attn_q").T).view(T, w.n_heads, hd).transpose(0, 1)
    k = (th @ W(f"{p}.attn_k").T).view(T, w.n_kv_heads, hd).transpose(0, 1)
    v = (th @ W(f"{p}.attn_v").T).view(T, w.n_kv_heads, hd).transpose(0, 1)
    gq = torch.from_numpy(m.gain(f"{p}.attn_q_norm"))
    gk = torch.from_numpy(m.gain(f"{p}.attn_k_norm"))
    q = rot(F.rms_norm(q, (hd,), weight=gq, eps=w.rms_eps))
    k16 = rot(F.rms_norm(k, (hd,), weight=gk, eps=w.rms_eps)).half().double()
    v16 = v.half().double()
    ck, cv = cache[0]
    assert np.array_equal(ck, k16.numpy()) and np.array_equal(cv, v16.numpy())
    o = F.scaled_dot_product_attention(q, k16.repeat_interleave(w.group, 0),
                                       v16.repeat_interleave(w.group, 0), is_causal=True)
    ref = (o.transpose(0, 1).reshape(T, -1) @ W(f"{p}.attn_output").T).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- sampling

def test_top_p_hand_worked():
    from oracle import sample as osm
    g = golden("sample_top_p.txt")
    probs = np.array([float(v) for v in g["probs"][0]])
    logits = np.log(probs)
    top_p = float(g["top_p"][0][0])
    order, q = osm.nucleus(logits, 1.0, top_p)
    assert order.tolist() == [int(v) for v in g["kept"][0]]
    assert np.allclose(q, np.array([0.5, 0.3, 0.15]) / 0.95, rtol=0, atol=1e-12)
    for u, tok in g["draw"]:
        assert osm.sample(logits, 1.0, top_p, float(u)) == int(tok), u
    small = float(g["top_p_small"][0][0])
    for u, tok in g["draw_small"]:
        assert osm.sample(logits, 1.0, small, float(u)) == int(tok)


def test_sampling_special_cases():
    """Temperature 0 is the argmax; top_p = 1 keeps every token and the draw
    follows the brute-force inverse CDF of the tempered softmax; a higher
    temperature flattens the distribution; equal logits draw in index order."""
    from oracle import sample as osm
    rng = np.random.default_rng(3)
    logits = rng.standard_normal(50) * 2.0
    assert osm.sample(logits, 0.0, 0.95, 0.7) == int(np.argmax(logits))
    T = 0.7
    p = np.exp(logits / T - np.max(logits / T))
    p /= p.sum()
    order = sorted(range(50), key=lambda i: (-p[i], i))    # brute force, plain Python
    for u in np.linspace(0.0, 0.999, 37):
        acc, pick = 0.0, order[-1]
        for i in order:
            acc += p[i]
            if acc > u:
                pick = i
                break
        assert osm.sample(logits, T, 1.0, float(u)) == pick, u
    o1, q1 = osm.nucleus(logits, 0.5, 1.0)
    o2, q2 = osm.nucleus(logits, 2.0, 1.0)
    assert q1[0] > q2[0]                                    # colder: a sharper top token
    eq = np.zeros(6)
    assert [osm.sample(eq, 1.0, 1.0, u) for u in (0.0, 0.2, 0.4, 0.6, 0.8, 0.95)] == [0, 1, 2, 3, 4, 5]
    o, q = osm.nucleus(eq, 1.0, 0.5)                        # ties kept in index order
    assert o.tolist() == [0, 1, 2] and np.allclose(q, 1 / 3)


# --------------------------------------------------------------------------- sibling architectures

def test_gelu_tanh_matches_torch_and_is_not_exact_gelu():
    z = np.linspace(-12, 12, 4001)
    ref = F.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    assert np.allclose(om.gelu_tanh(z), ref, rtol=1e-14, atol=1e-15)
    exact = F.gelu(torch.from_numpy(z)).numpy()
    gap = np.max(np.abs(om.gelu_tanh(z) - exact))
    assert 1e-5 < gap < 2e-3           # two different functions, ~1e-3 apart at most
    assert om.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert np.isclose(om.gelu_tanh(np.array([30.0]))[0], 30.0, rtol=0, atol=1e-12)


def test_softcap_closed_form():
    c = 30.0
    x = np.array([-1e4, -30.0, -1e-3, 0.0, 1e-3, 30.0, 1e4])
    y = om.softcap(x, c)
    assert np.allclose(y, c * torch.tanh(torch.from_numpy(x) / c).numpy(), rtol=1e-15)
    assert np.isclose(y[0], -c) and np.isclose(y[-1], c)                  # saturates at +-c
    assert np.isclose(y[4], 1e-3, rtol=1e-9) and y[3] == 0.0             # identity near 0
    assert np.isclose(y[5], c * math.tanh(1.0), rtol=1e-15)
    r = np.random.default_rng(1).standard_normal(1000) * 50
    assert np.all(np.diff(om.softcap(np.sort(r), c)) >= 0)               # order kept: argmax unchanged


@pytest.mark.parametrize("window", [1, 3, 5, 13, 40])
def test_sliding_window_attention_matches_sdpa_band_mask(window):
    rng = np.random.default_rng(window)
    nq, nkv, T, hd = 4, 2, 13, 16
    q, k, v = (rng.standard_normal((n, T, hd)) for n in (nq, nkv, nkv))
    pos = np.arange(T)
    out = om.attention(q, k, v, pos, window)
    j, p = np.arange(T)[None, :], pos[:, None]
    band = torch.from_numpy((j <= p) & (j > p - window))
    G = nq // nkv
    ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k).repeat_interleave(G, 0),
                                         torch.from_numpy(v).repeat_interleave(G, 0), attn_mask=band).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)
    if window >= T:
        assert np.allclose(out, om.attention(q, k, v, pos), rtol=0, atol=0)
    if window == 1:  # each query sees only its own key: the output is that key's value row
        assert np.allclose(out, np.repeat(v, G, axis=0), rtol=1e-13)


def _tiny_arch(arch, kv="f32"):
    w = synth.Workload("pin_" + arch, vocab=512, hidden=128, n_layers=4, n_heads=4, n_kv_heads=2,
                       head_dim=32, ffn=256, wtype="q8_0", kv=kv, seed=0, arch=arch,
                       sliding_window=3 if arch == "gemma3" else 0, sliding_pattern=2,
                       logit_softcap=0.5 if arch == "gemma3" else 0.0)
    return w, om.OracleModel(w, om.synth_weights(w))


@pytest.mark.parametrize("arch", ["llama", "qwen2", "gemma3", "qwen3"])
def test_arch_models_match_torch_library_composition(arch):
    """Each layer recipe recomposed from torch library routines: F.rms_norm,
    bias adds, SDPA with a band mask for sliding layers, F.gelu(approximate=
    "tanh") or F.silu, torch.tanh for the softcap."""
    w, m = _tiny_arch(arch)
    prompt = list(w.prompt(n=9))
    T, hd = len(prompt), w.head_dim

    def W(n):
        return torch.from_numpy(m.matrix(n))

    def g(n):
        return torch.from_numpy(np.asarray(m.weights[n], dtype=np.float32).astype(np.float64))

    x = torch.from_numpy(m.embed(prompt))
    pos = np.arange(T)
    ang = torch.from_numpy(om.rope_angles(pos, hd, w.rope_theta))
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rot(t):
        a, b = t[..., : hd // 2], t[..., hd // 2:]
        return torch.cat([a * cos - b * sin, a * sin + b * cos], -1)

    for i in range(w.n_layers):
        p = f"blk.{i}"
        h = F.rms_norm(x, (w.hidden,), weight=g(f"{p}.attn_norm"), eps=w.rms_eps)
        q, k, v = h @ W(f"{p}.attn_q").T, h @ W(f"{p}.attn_k").T, h @ W(f"{p}.attn_v").T
        if arch == "qwen2":
            q, k, v = q + g(f"{p}.attn_q_bias"), k + g(f"{p}.attn_k_bias"), v + g(f"{p}.attn_v_bias")
        q = q.view(T, w.n_heads, hd).transpose(0, 1)
        k = k.view(T, w.n_kv_heads, hd).transpose(0, 1)
        v = v.view(T, w.n_kv_heads, hd).transpose(0, 1)
        if arch in ("qwen3", "gemma3"):
            q = F.rms_norm(q, (hd,), weight=g(f"{p}.attn_q_norm"), eps=w.rms_eps)
            k = F.rms_norm(k, (hd,), weight=g(f"{p}.attn_k_norm"), eps=w.rms_eps)
        q, k = rot(q), rot(k)
        sliding = arch == "gemma3" and i % 2 == 0      # pattern 2: odd layers are global
        j, pp = torch.arange(T)[None, :], torch.arange(T)[:, None]
        mask = (j <= pp) & ((j > pp - 3) if sliding else True)
        o = F.scaled_dot_product_attention(q, k.repeat_interleave(w.group, 0), v.repeat_interleave(w.group, 0),
                                           attn_mask=mask)
        x = x + o.transpose(0, 1).reshape(T, -1) @ W(f"{p}.attn_output").T
        h = F.rms_norm(x, (w.hidden,), weight=g(f"{p}.ffn_norm"), eps=w.rms_eps)
        gate = h @ W(f"{p}.ffn_gate").T
        act = F.gelu(gate, approximate="tanh") if arch == "gemma3" else F.silu(gate)
        x = x + (act * (h @ W(f"{p}.ffn_up").T)) @ W(f"{p}.ffn_down").T
    xl = F.rms_norm(x[-1], (w.hidden,), weight=g("output_norm"), eps=w.rms_eps)
    ref = xl @ W("token_embd").T
    if arch == "gemma3":
        ref = 0.5 * torch.tanh(ref / 0.5)
    assert np.allclose(m.forward_nocache(prompt), ref.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("arch", ["llama", "qwen2", "gemma3"])
def test_arch_cached_decode_equals_full_recompute(arch):
    """The KV cache (and the sliding window on it) gives the same logits as
    rebuilding the prefix with no state, every step."""
    w, m = _tiny_arch(arch)
    prompt = list(w.prompt(n=5))
    toks, logits = om.run_greedy(m, prompt, 6)
    seq = prompt + toks[:-1]
    for s in range(7):
        ref = m.forward_nocache(seq[: len(prompt) + s])
        assert np.allclose(logits[s], ref, rtol=1e-12, atol=1e-12), s


# --------------------------------------------------------------------------- affine 4-bit format

def _golden_affine():
    return {k: v[0] for k, v in golden("affine4_group.txt").items()}


def test_affine4_hand_worked_group():
    rec = _golden_affine()
    w = np.zeros(64, dtype=np.float32)
    w[:5] = [float(v) for v in rec["values"]]
    g = quant.quantize_affine4(w[None, :])[0, 0]
    words = g[0:32].copy().view("<u4")
    assert int(words[0]) == int(rec["word0"][0], 16)
    assert all(int(x) == int(rec["word_rest"][0], 16) for x in words[1:])
    assert int(g[32:34].copy().view("<u2")[0]) == int(rec["scale_bf16"][0], 16)
    assert int(g[34:36].copy().view("<u2")[0]) == int(rec["bias_bf16"][0], 16)
    q, _, _ = quant.affine4_parts(g[None, :])
    assert q[0, :5].tolist() == [int(v) for v in rec["codes"]]
    deq = quant.dequantize(g[None, None, :], "affine4")[0]
    assert deq[:5].tolist() == [float(v) for v in rec["decoded"]]
    assert np.all(deq[5:] == 0.0)


def test_affine4_brute_force_error_bound_and_equal_groups():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((7, 256)) * 0.02).astype(np.float32)
    w[3, 64:128] = 0.0375                                  # a group of equal values
    g = quant.quantize_affine4(w)
    q, sb, bb = quant.affine4_parts(g)
    deq = quant.dequantize(g, "affine4").reshape(7, 4, 64)
    grp = w.astype(np.float64).reshape(7, 4, 64)
    lo, hi = grp.min(-1), grp.max(-1)
    s = (hi - lo) / 15
    s_bf, b_bf = quant.bf16_value(sb).astype(np.float64), quant.bf16_value(bb).astype(np.float64)
    bound = s / 2 + 15 * np.abs(s - s_bf) + np.abs(lo - b_bf) + 1e-9
    assert np.all(np.abs(deq - grp) <= bound[..., None])
    assert q[3, 1].max() == 0 and s_bf[3, 1] == 0.0 and np.all(deq[3, 1] == b_bf[3, 1])
    # codes in range, extremes hit
    assert q.max() == 15 and q.min() == 0
    # decoding in f32 rounds once: within half an ulp of the f64 value
    d32 = quant.dequantize(g, "affine4", np.float32).astype(np.float64).reshape(7, 4, 64)
    assert np.all(np.abs(d32 - deq) <= np.abs(deq) * 2.0 ** -24 + 1e-30)
