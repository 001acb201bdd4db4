"""GPU parity of batched decode: several sequences of different lengths in one
tq_decode_step, over the contiguous cache (sequence b in slot b) and over a
paged cache whose pages are handed out in a shuffled order, each sequence
against its own oracle run (teacher-forced on the oracle's greedy tokens).
Tolerances as in test_gpu_model: 2e-3 of the oracle's logit range with an f32
KV cache, 1e-2 with f16."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import model as om
from block_quantized_transformer_gb300.synthetic import build_model
from gpu_util import rel_logit_err, check_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _oracle_runs(w, lens, steps):
    ref = om.OracleModel(w, om.synth_weights(w))
    runs = []
    for b, n in enumerate(lens):
        prompt = list(w.prompt(b, n=n))
        toks, logits = om.run_greedy(ref, prompt, steps)
        runs.append((prompt, toks, logits))
    return runs


def _batched_case(w, lens, steps, page_size=0, n_pages=0, seed=7):
    B = len(lens)
    max_ctx = 64
    runs = _oracle_runs(w, lens, steps)
    model = build_model(w, device=DEV, max_batch=B, max_ctx=max_ctx, max_prefill=max(lens),
                        page_size=page_size, n_pages=n_pages)
    V = w.vocab
    tol = 2e-3 if w.kv == "f32" else 1e-2
    bt = None
    if page_size:
        per_seq = max_ctx // page_size
        perm = np.random.RandomState(seed).permutation(n_pages)[:B * per_seq]
        bt = torch.tensor(perm.reshape(B, per_seq), dtype=torch.int32, device=DEV)
    got = [[] for _ in range(B)]
    got_tok = [[] for _ in range(B)]
    for b, (prompt, _, _) in enumerate(runs):
        lg = torch.empty(V, dtype=torch.float32, device=DEV)
        am = model.prefill(torch.tensor(prompt, dtype=torch.int32, device=DEV), seq=b,
                           block_table=None if bt is None else bt[b].contiguous(), logits=lg)
        got[b].append(lg.double().cpu().numpy())
        got_tok[b].append(int(am.item()))
    for s in range(steps):
        toks = torch.tensor([runs[b][1][s] for b in range(B)], dtype=torch.int32, device=DEV)
        pos = torch.tensor([lens[b] + s for b in range(B)], dtype=torch.int32, device=DEV)
        lg = torch.empty(B, V, dtype=torch.float32, device=DEV)
        am = model.decode_step(toks, pos, pos.clone(), block_table=bt, logits=lg)
        for b in range(B):
            got[b].append(lg[b].double().cpu().numpy())
            got_tok[b].append(int(am[b].item()))
    assert model.status() == 0
    model.close()
    for b in range(B):
        ref_logits = runs[b][2]
        errs = [rel_logit_err(g, r) for g, r in zip(got[b], ref_logits)]
        assert max(errs) <= tol, (b, max(errs), int(np.argmax(errs)))
        check_tokens(got_tok[b], ref_logits, tol)


def test_batched_decode_contiguous_cache():
    _batched_case(synth.TINY, [5, 12, 9], steps=6)


def test_batched_decode_paged_ragged():
    # 37 + 10 > 32: sequences cross page boundaries; pages are shuffled
    _batched_case(synth.TINY, [20, 37, 50, 3], steps=10, page_size=32, n_pages=11)


def test_batched_decode_paged_f16_q4_0():
    w = dataclasses.replace(synth.TINY, wtype="q4_0", kv="f16")
    _batched_case(w, [33, 7], steps=8, page_size=32, n_pages=5, seed=3)


def test_batched_decode_split_k_projections():
    # hidden 1024 / ffn 3072: every projection has 4-12 K units and few CTAs
    # at 4 rows, so the GEMMs split K across CTAs and add the partial sums
    w = dataclasses.replace(synth.TINY, name="split_k_q4_0", hidden=1024, ffn=3072, n_heads=8,
                            n_kv_heads=4, head_dim=128, wtype="q4_0", kv="f16")
    _batched_case(w, [9, 4, 17, 12], steps=4, page_size=32, n_pages=9, seed=5)


def test_batched_decode_split_k_q8_0():
    # the split-K GEMM of the Q8_0 kernel (one CTA per SM), contiguous f32 cache
    w = dataclasses.replace(synth.TINY, name="split_k_q8_0", hidden=1024, ffn=3072, n_heads=8,
                            n_kv_heads=4, head_dim=128, wtype="q8_0", kv="f32")
    _batched_case(w, [6, 15, 3], steps=3)


def test_batched_decode_paged_f16_group_of_8():
    # 4-CTA tensor-core attention clusters with two n-tiles (8 query heads per KV head)
    w = dataclasses.replace(synth.TINY, name="batched_g8", hidden=512, n_heads=8, n_kv_heads=1, kv="f16")
    _batched_case(w, [18, 41, 7], steps=5, page_size=32, n_pages=7, seed=11)
