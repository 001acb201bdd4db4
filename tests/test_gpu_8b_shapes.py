"""GPU parity at the Qwen3-8B shape (hidden 4096, 32 query / 8 KV heads,
head_dim 128, FFN 12288, vocab 151936, Q4_0, f16 KV) with two of its 36 layers:
the kernel instantiations the benchmarked workloads launch (tensor-core
attention with 4 query heads per KV head in its fused 16-CTA decode mode, its
4-CTA batched mode and its non-fused prefill mode; the Q4_0 GEMMs at K = 4096
and 12288; the 151936-row head), against the oracle in float32 on the same
seeded weights.

* batch 1: the full 2048-token prompt, then 16 decode steps teacher-forced on
  the oracle's greedy tokens;
* batched: the 32 ragged context lengths of the batched serving mix (seeded,
  512..8192) over a paged cache of 64-token pages handed out in a seeded
  shuffled order; the cached K/V are seeded f16 values written identically to
  both sides (the pages do not say what the contexts hold), then 4 batched
  decode steps, each sequence teacher-forced on its own oracle run.

Tolerance (f16 KV): max |logit error| / oracle logit range <= 1e-2 per step;
greedy tokens equal wherever the oracle's top-2 margin exceeds that."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import model as om
from block_quantized_transformer_gb300.synthetic import build_model, build_weights
from gpu_util import rel_logit_err, check_tokens, gpu_teacher_forced

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 1e-2
W1 = dataclasses.replace(synth.QWEN3_8B_Q4, name="qwen3_8b_q4_0_2layers", n_layers=2)
WB = dataclasses.replace(synth.QWEN3_8B_Q4_BATCHED, name="qwen3_8b_q4_0_batched32_2layers", n_layers=2)


@pytest.fixture(scope="module")
def weights():
    """Oracle block bytes (host) and GPU tiled weights (device) of the 2-layer
    8B-shaped model; the batched workload has the same seed and shapes."""
    assert (WB.seed, WB.hidden, WB.ffn, WB.vocab) == (W1.seed, W1.hidden, W1.ffn, W1.vocab)
    host = om.synth_weights(W1)
    dev = build_weights(W1, DEV)
    torch.cuda.synchronize()
    return host, dev


def test_qwen3_8b_shape_batch1_2048_prompt(weights):
    host, dev = weights
    steps = 16
    prompt = list(W1.prompt(n=W1.prompt_len))
    ref = om.OracleModel(W1, host, dtype=np.float32)
    toks, ref_logits = om.run_greedy(ref, prompt, steps)
    model = build_model(W1, device=DEV, max_ctx=len(prompt) + steps + 1, max_prefill=len(prompt),
                        weights=dev)
    got_l, got_t = gpu_teacher_forced(model, prompt, toks[:steps], DEV)
    assert model.status() == 0
    model.close()
    errs = [rel_logit_err(g, r) for g, r in zip(got_l, ref_logits)]
    print(f"8B-shape batch 1: max rel logit err {max(errs):.3e} (prefill {errs[0]:.3e})")
    assert max(errs) <= TOL, (max(errs), int(np.argmax(errs)))
    assert check_tokens(got_t, ref_logits, TOL) >= 0.5 * len(got_t)


def _page_table(lens, extra, P):
    """Pages of each sequence (enough for its context plus `extra` tokens),
    drawn from one pool in a seeded shuffled order."""
    n_seq_pages = (lens + extra + P - 1) // P
    n_pages = int(n_seq_pages.sum())
    keys = synth.host_normal(WB.length_seed, synth.LENGTH_STREAM + 1, n_pages, sigma=1.0)
    order = np.argsort(keys, kind="stable").astype(np.int32)
    per_seq = int(n_seq_pages.max())
    table = np.zeros((len(lens), per_seq), dtype=np.int32)
    at = 0
    for b, n in enumerate(n_seq_pages):
        table[b, :n] = order[at:at + n]
        at += n
    return table, n_pages, per_seq


def _seeded_contexts(lens, table, n_pages):
    """Seeded f16 K/V of every cached position, written identically to the
    paged device layout [layer][page][kv head][slot][hd] (host tensors) and to
    the oracle's per-sequence caches ([layer] -> (K, V) of [nkv][len][hd])."""
    w = WB
    B, P, L, nkv, hd = w.batch, w.page_size, w.n_layers, w.n_kv_heads, w.head_dim
    caches = []
    kc = torch.zeros(L, n_pages, nkv, P, hd, dtype=torch.float16)
    vc = torch.zeros(L, n_pages, nkv, P, hd, dtype=torch.float16)
    for b in range(len(lens)):
        n = int(lens[b])
        npg = (n + P - 1) // P
        per_layer = []
        for l in range(L):
            kv = []
            for j, dst in enumerate((kc, vc)):
                stream = synth.KV_STREAM + 2 * (l * B + b) + j
                x = synth.host_normal(w.seed, stream, nkv * n * hd, sigma=1.0).astype(np.float16)
                x = x.reshape(nkv, n, hd)
                kv.append(x.astype(np.float32))
                if n == 0:
                    continue
                pad = np.zeros((nkv, npg * P, hd), dtype=np.float16)
                pad[:, :n] = x
                pages = torch.from_numpy(pad.reshape(nkv, npg, P, hd).transpose(1, 0, 2, 3).copy())
                dst[l, torch.from_numpy(table[b, :npg]).long()] = pages
            per_layer.append((kv[0], kv[1]))
        caches.append(per_layer)
    return kc, vc, caches


def test_qwen3_8b_shape_batched32_paged_ragged(weights):
    host, dev = weights
    steps = 4
    w = WB
    B, P, L, nkv, hd = w.batch, w.page_size, w.n_layers, w.n_kv_heads, w.head_dim
    lens = w.context_lengths().astype(np.int64)
    assert len(lens) == 32 and lens.min() >= 512 and lens.max() <= 8192
    table, n_pages, per_seq = _page_table(lens, steps + 1, P)

    kc, vc, caches = _seeded_contexts(lens, table, n_pages)

    # oracle: each sequence on its own cache, greedy from a seeded first token
    ref = om.OracleModel(w, host, dtype=np.float32)
    first = synth.uniform_below(w.seed, synth.PROMPT_STREAM, B, w.vocab)
    feed = [[int(first[b])] for b in range(B)]
    ref_logits = [[] for _ in range(B)]
    for s in range(steps):
        for b in range(B):
            lg = ref.forward([feed[b][s]], caches[b], int(lens[b]) + s)
            ref_logits[b].append(lg)
            feed[b].append(om.argmax(lg))

    model = build_model(w, device=DEV, max_batch=B, max_ctx=per_seq * P, max_prefill=B,
                        page_size=P, n_pages=n_pages, weights=dev)
    model.k_cache.copy_(kc.reshape(-1))
    model.v_cache.copy_(vc.reshape(-1))
    del kc, vc
    bt = torch.from_numpy(table).to(DEV)
    got_l = [[] for _ in range(B)]
    got_t = [[] for _ in range(B)]
    for s in range(steps):
        tok = torch.tensor([feed[b][s] for b in range(B)], dtype=torch.int32, device=DEV)
        pos = torch.tensor((lens + s).astype(np.int32), device=DEV)
        lg = torch.empty(B, w.vocab, dtype=torch.float32, device=DEV)
        am = model.decode_step(tok, pos, pos.clone(), block_table=bt, logits=lg)
        lg_h, am_h = lg.double().cpu().numpy(), am.cpu().numpy()
        for b in range(B):
            got_l[b].append(lg_h[b])
            got_t[b].append(int(am_h[b]))
    assert model.status() == 0
    model.close()
    worst = 0.0
    for b in range(B):
        errs = [rel_logit_err(g, r) for g, r in zip(got_l[b], ref_logits[b])]
        worst = max(worst, max(errs))
        assert max(errs) <= TOL, (b, int(lens[b]), max(errs), int(np.argmax(errs)))
        check_tokens(got_t[b], ref_logits[b], TOL)
    print(f"8B-shape batched 32 paged: max rel logit err {worst:.3e}")


def test_qwen3_8b_shape_mixed_step_paged(weights):
    """Continuous batching at the 8B shape: one tq_step over 8 decode rows of
    the batched mix's first 8 sequences, a 249-row prompt chunk of a sequence
    with 320 cached positions and a 40-row prompt from position 0 (297 rows:
    the GEMMs take two 256-row token tiles, the second ragged), then one step
    in which all 10 sequences decode; each sequence's rows are compared with
    the oracle running that sequence alone on the same cache."""
    host, dev = weights
    w = WB
    P = w.page_size
    dec = w.context_lengths().astype(np.int64)[:8]
    chunk_a, cached_a, chunk_b = 249, 320, 40
    lens = np.concatenate([dec, [cached_a, 0]]).astype(np.int64)
    S = len(lens)
    table, n_pages, per_seq = _page_table(lens, chunk_a + 2, P)
    kc, vc, caches = _seeded_contexts(lens, table, n_pages)
    first = synth.uniform_below(w.seed, synth.PROMPT_STREAM + 100, S, w.vocab)
    feeds = [[int(first[b])] for b in range(8)]
    feeds.append(list(synth.uniform_below(w.seed, synth.PROMPT_STREAM + 101, chunk_a, w.vocab)))
    feeds.append(list(synth.uniform_below(w.seed, synth.PROMPT_STREAM + 102, chunk_b, w.vocab)))

    ref = om.OracleModel(w, host, dtype=np.float32)
    ref_l = [[] for _ in range(S)]
    nxt = []
    for b in range(S):
        lg = ref.forward(feeds[b], caches[b], int(lens[b]))
        ref_l[b].append(lg)
        nxt.append(om.argmax(lg))
    for b in range(S):                                 # step 2: every sequence decodes its greedy token
        ref_l[b].append(ref.forward([nxt[b]], caches[b], int(lens[b]) + len(feeds[b])))

    n_rows = sum(len(f) for f in feeds)
    model = build_model(w, device=DEV, max_batch=S, max_ctx=per_seq * P, max_prefill=n_rows,
                        page_size=P, n_pages=n_pages, weights=dev)
    model.k_cache.copy_(kc.reshape(-1))
    model.v_cache.copy_(vc.reshape(-1))
    del kc, vc
    bt = torch.from_numpy(table).to(DEV)
    got_l = [[] for _ in range(S)]
    got_t = [[] for _ in range(S)]
    steps = [[(b, feeds[b], int(lens[b])) for b in range(S)],
             [(b, [nxt[b]], int(lens[b]) + len(feeds[b])) for b in range(S)]]
    for rows in steps:
        tok, seq, pos, last = [], [], [], []
        for b, toks, p0 in rows:
            tok += [int(t) for t in toks]
            seq += [b] * len(toks)
            pos += list(range(p0, p0 + len(toks)))
            last.append(len(tok) - 1)
        i32 = lambda v: torch.tensor(v, dtype=torch.int32, device=DEV)
        lg = torch.empty(S, w.vocab, dtype=torch.float32, device=DEV)
        am = model.step(i32(tok), i32(seq), i32(pos), i32(last), block_table=bt, logits=lg)
        lg_h, am_h = lg.double().cpu().numpy(), am.cpu().numpy()
        for b in range(S):
            got_l[b].append(lg_h[b])
            got_t[b].append(int(am_h[b]))
    assert model.status() == 0
    model.close()
    worst = 0.0
    for b in range(S):
        errs = [rel_logit_err(g, r) for g, r in zip(got_l[b], ref_l[b])]
        worst = max(worst, max(errs))
        assert max(errs) <= TOL, (b, int(lens[b]), max(errs), int(np.argmax(errs)))
        check_tokens(got_t[b], ref_l[b], TOL)
    print(f"8B-shape mixed step ({n_rows} rows, {S} sequences): max rel logit err {worst:.3e}")
