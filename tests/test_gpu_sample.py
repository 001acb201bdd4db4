"""GPU parity of temperature / top-p sampling (tq_sample) against the oracle's
sampler on the same logits and uniform numbers.  The token is an integer
decided by f32 sums on the GPU and f64 in the oracle, so a draw is compared
exactly wherever u and top_p sit more than 1e-5 (in probability) from the
cumulative sums that decide it; otherwise (over 151936 tokens of a flat
distribution the sums are closer together than f32 resolves) the drawn token
must lie in the oracle's kept set, with its interval of the oracle's
cumulative distribution within 1e-4 of u."""
import numpy as np
import pytest
import torch

import synth
from oracle import sample as osm
import block_quantized_transformer_gb300 as tq

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(logits, temps, top_ps, us):
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(DEV)
    t = torch.tensor(temps, dtype=torch.float32, device=DEV)
    p = torch.tensor(top_ps, dtype=torch.float32, device=DEV)
    u = torch.tensor(us, dtype=torch.float32, device=DEV)
    return tq.tq_sample(lg, t, p, u).cpu().numpy()


def _check(logits, temps, top_ps, us, min_exact, rows_per_call=None):
    k = rows_per_call or len(temps)
    got = np.concatenate([_run(logits[i:i + k], temps[i:i + k], top_ps[i:i + k], us[i:i + k])
                          for i in range(0, len(temps), k)])
    exact = 0
    for r in range(len(temps)):
        row = logits[r].astype(np.float64)
        ref = osm.sample(row, temps[r], top_ps[r], us[r])
        if temps[r] == 0:
            assert got[r] == ref, (r, got[r], ref)
            exact += 1
            continue
        if osm.boundary_distance(row, temps[r], top_ps[r], us[r]) > 1e-5:
            assert got[r] == ref, (r, temps[r], top_ps[r], us[r], got[r], ref)
            exact += 1
        else:
            kept, q = osm.nucleus(row, temps[r], top_ps[r])
            pos = {int(t): k for k, t in enumerate(kept)}
            assert int(got[r]) in pos, (r, got[r])
            k = pos[int(got[r])]
            lo, hi = float(np.sum(q[:k])), float(np.sum(q[:k + 1]))
            assert lo - 1e-4 <= us[r] <= hi + 1e-4, (r, us[r], lo, hi)
    assert exact >= min_exact, exact


def test_sample_vocab_151936_matches_oracle():
    V, n = 151936, 48
    base = synth.host_normal(11, 1, 4 * V, sigma=1.0).reshape(4, V)
    base[1] *= 3.0                                    # a sharper distribution
    base[3] = np.round(base[3] * 4.0) / 4.0           # many exactly equal logits
    logits = np.repeat(base, n // 4, axis=0)
    us = synth.uniform_below(11, 2, n, 1 << 24).astype(np.float64) / float(1 << 24)
    temps = [[0.0, 0.7, 1.0, 1.6][i % 4] for i in range(n)]
    top_ps = [[0.95, 0.5, 1.0, 0.9, 0.05, 0.99][i % 6] for i in range(n)]
    _check(logits, temps, top_ps, list(us), min_exact=16)


@pytest.mark.parametrize("rows_per_call", [1, 8, 32])
def test_sample_vocab_151936_per_call_batch(rows_per_call):
    """The same rows sampled 1, 8 and 32 to a call: one row is split across a
    cluster of up to 16 CTAs, 32 rows across 4 each."""
    V = 151936
    n = 32 if rows_per_call > 1 else 8
    base = synth.host_normal(11, 1, 4 * V, sigma=1.0).reshape(4, V)
    base[1] *= 3.0
    base[3] = np.round(base[3] * 4.0) / 4.0
    logits = np.repeat(base, n // 4, axis=0)
    us = synth.uniform_below(11, 5, n, 1 << 24).astype(np.float64) / float(1 << 24)
    temps = [[0.0, 0.7, 1.0, 1.6][i % 4] for i in range(n)]
    top_ps = [[0.95, 0.5, 1.0, 0.9, 0.05, 0.99][i % 6] for i in range(n)]
    _check(logits, temps, top_ps, list(us), min_exact=n // 3, rows_per_call=rows_per_call)


def test_sample_small_vocab_and_ties():
    # all logits equal: the draw walks the tokens in index order
    eq = np.zeros((6, 7), dtype=np.float32)
    us = [0.0, 0.15, 0.3, 0.5, 0.75, 0.99]
    got = _run(eq, [1.0] * 6, [1.0] * 6, us)
    assert got.tolist() == [int(u * 7) for u in us]
    # top_p keeps the first ceil(top_p * 7) of them
    got = _run(eq[:3], [1.0] * 3, [0.3] * 3, [0.0, 0.5, 0.99])
    assert got.tolist() == [0, 1, 2]
    # greedy with a planted tie: the lower index
    row = np.array([[0.5, 2.0, -1.0, 2.0, 1.9]], dtype=np.float32)
    assert _run(row, [0.0], [0.9], [0.3]).tolist() == [1]
    # random small rows against the oracle
    rng_logits = synth.host_normal(12, 3, 64 * 33, sigma=2.0).reshape(64, 33)
    us = synth.uniform_below(12, 4, 64, 1 << 24).astype(np.float64) / float(1 << 24)
    _check(rng_logits, [0.8] * 64, [0.9] * 64, list(us), min_exact=56)


def test_sample_temperature_zero_equals_decode_argmax():
    from block_quantized_transformer_gb300.synthetic import build_model
    w = synth.TINY
    m = build_model(w, device=DEV, max_ctx=32)
    prompt = torch.tensor(w.prompt(), dtype=torch.int32, device=DEV)
    am = m.prefill(prompt)
    tok = am.clone()
    p = torch.tensor([len(prompt)], dtype=torch.int32, device=DEV)
    lg = torch.empty(1, w.vocab, device=DEV)
    am2 = m.decode_step(tok, p, p, logits=lg)
    t0 = torch.zeros(1, device=DEV)
    got = tq.tq_sample(lg, t0, torch.ones(1, device=DEV), torch.zeros(1, device=DEV))
    assert int(got.item()) == int(am2.item())
    m.close()
