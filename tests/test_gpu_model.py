"""End-to-end GPU parity of the decode step: the GPU model (device-generated
weights, GPU encoder, tiled repack, all kernels) against the oracle on the
same seeded inputs, teacher-forced on the oracle's greedy tokens.  Tolerance:
max |logit error| / oracle logit range <= 2e-3 with an f32 KV cache, 1e-2
with f16; greedy tokens equal wherever the oracle's top-2 margin exceeds that
tolerance times the range."""
import numpy as np
import pytest
import torch

import synth
from oracle import model as om
from block_quantized_transformer_gb300.synthetic import build_model
from gpu_util import rel_logit_err, check_tokens, gpu_teacher_forced

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def tol_of(w):
    return 2e-3 if w.kv == "f32" else 1e-2


def run_case(w, prompt_len, steps, graph=False):
    prompt = list(w.prompt(n=prompt_len))
    ref = om.OracleModel(w, om.synth_weights(w))
    toks, ref_logits = om.run_greedy(ref, prompt, steps)
    model = build_model(w, device=DEV, max_ctx=prompt_len + steps + 1, max_prefill=prompt_len)
    got_l, got_t = gpu_teacher_forced(model, prompt, toks[:steps], DEV)
    assert model.status() == 0
    tol = tol_of(w)
    errs = [rel_logit_err(g, r) for g, r in zip(got_l, ref_logits)]
    assert max(errs) <= tol, (max(errs), int(np.argmax(errs)))
    n = check_tokens(got_t, ref_logits, tol)
    assert n >= 0.5 * len(got_t)
    model.close()
    return errs


def test_tiny_q8_0_full_workload():
    w = synth.TINY
    errs = run_case(w, w.prompt_len, w.decode_steps)
    print(f"tiny Q8_0: max rel logit err {max(errs):.3e} (prefill {errs[0]:.3e})")


def test_tiny_variants_f16_kv_and_q4_0():
    import dataclasses
    for wt, kv in [("q4_0", "f16"), ("q8_0", "f16"), ("q4_0", "f32")]:
        w = dataclasses.replace(synth.TINY, name=f"tiny_{wt}_{kv}", wtype=wt, kv=kv)
        run_case(w, 13, 9)


def test_tiny_gqa_group_sizes():
    import dataclasses
    for nq, nkv in [(4, 4), (8, 1), (8, 2)]:
        w = dataclasses.replace(synth.TINY, name=f"tiny_g{nq // nkv}", n_heads=nq, n_kv_heads=nkv,
                                hidden=512)
        run_case(w, 11, 5)


def test_prefill_in_chunks_equals_one_shot():
    w = synth.TINY
    prompt = torch.tensor(w.prompt(n=40), dtype=torch.int32, device=DEV)
    a = build_model(w, device=DEV, max_ctx=64, max_prefill=40)
    la = torch.empty(w.vocab, device=DEV)
    a.prefill(prompt, logits=la)
    b = build_model(w, device=DEV, max_ctx=64, max_prefill=40)
    lb = torch.empty(w.vocab, device=DEV)
    b.prefill(prompt[:17], logits=lb)
    b.prefill(prompt[17:], start_pos=17, logits=lb)
    assert torch.allclose(la, lb, rtol=0, atol=1e-4 * float(la.max() - la.min()))


def test_graph_replay_equals_eager():
    w = synth.TINY
    prompt = torch.tensor(w.prompt(), dtype=torch.int32, device=DEV)
    outs = []
    for graph in (False, True):
        m = build_model(w, device=DEV, max_ctx=32)
        s = torch.cuda.Stream(device=DEV)
        with torch.cuda.stream(s):
            am = m.prefill(prompt)
            tok = torch.empty(1, dtype=torch.int32, device=DEV)
            pos = torch.empty(1, dtype=torch.int32, device=DEV)
            lg = torch.empty(1, w.vocab, device=DEV)
            seq = []
            tok.copy_(am)
            for st in range(6):
                pos.fill_(len(prompt) + st)
                am2 = torch.empty(1, dtype=torch.int32, device=DEV)
                m.decode_step(tok, pos, pos, logits=lg, argmax=am2, graph=graph)
                seq.append((int(am2.item()), lg.clone()))
                tok.copy_(am2)
        s.synchronize()
        outs.append(seq)
    for (t0, l0), (t1, l1) in zip(*outs):
        assert t0 == t1 and torch.equal(l0, l1)


def test_bad_token_sets_status_and_poisons():
    import block_quantized_transformer_gb300 as tq
    w = synth.TINY
    m = build_model(w, device=DEV, max_ctx=16)
    t = torch.tensor([w.vocab + 5], dtype=torch.int32, device=DEV)
    p = torch.tensor([0], dtype=torch.int32, device=DEV)
    m.decode_step(t, p, p)
    with pytest.raises(tq.TqPoisoned, match="token id out of range"):
        m.status()
    with pytest.raises(tq.TqError, match="closed"):
        m.decode_step(t, p, p)


def test_kv_overflow_is_refused_or_flagged():
    import block_quantized_transformer_gb300 as tq
    w = synth.TINY
    m = build_model(w, device=DEV, max_ctx=16, max_prefill=8)
    with pytest.raises(tq.TqError, match="exceeds max_ctx"):
        m.prefill(torch.zeros(8, dtype=torch.int32, device=DEV), start_pos=10)
    assert m.status() == 0                          # the refusal enqueued nothing
    p = torch.tensor([16], dtype=torch.int32, device=DEV)
    m.decode_step(torch.tensor([1], dtype=torch.int32, device=DEV), p, p)
    with pytest.raises(tq.TqPoisoned, match="out of range"):
        m.status()


def test_qwen3_0p6b_q8_0_full_workload():
    w = synth.QWEN3_0P6B_Q8
    errs = run_case(w, w.prompt_len, w.decode_steps)
    print(f"0.6B Q8_0: max rel logit err {max(errs):.3e} (prefill {errs[0]:.3e})")


def test_qwen3_0p6b_q4_0_long_context():
    # the whole workload: 4096-token prompt, then all 256 decode steps
    w = synth.QWEN3_0P6B_Q4_LONG
    errs = run_case(w, w.prompt_len, w.decode_steps)
    print(f"0.6B Q4_0 long context: max rel logit err {max(errs):.3e} over {len(errs)} steps")


def test_gqa_group_sizes_f16_cache():
    # the tensor-core attention (decode, and prefill in its non-fused mode) for
    # groups of 1, 8 and 4 query heads per KV head, head_dim 64
    import dataclasses
    for nq, nkv in [(4, 4), (8, 1), (8, 2)]:
        w = dataclasses.replace(synth.TINY, name=f"tiny_f16_g{nq // nkv}", n_heads=nq, n_kv_heads=nkv,
                                hidden=512, kv="f16")
        run_case(w, 11, 5)


def test_prefill_in_chunks_equals_one_shot_f16_cache():
    # the tensor-core prefill attention continues from a nonzero position
    import dataclasses
    w = dataclasses.replace(synth.TINY, name="tiny_f16_chunks", kv="f16")
    prompt = torch.tensor(w.prompt(n=40), dtype=torch.int32, device=DEV)
    a = build_model(w, device=DEV, max_ctx=64, max_prefill=40)
    la = torch.empty(w.vocab, device=DEV)
    a.prefill(prompt, logits=la)
    b = build_model(w, device=DEV, max_ctx=64, max_prefill=40)
    lb = torch.empty(w.vocab, device=DEV)
    b.prefill(prompt[:17], logits=lb)
    b.prefill(prompt[17:], start_pos=17, logits=lb)
    assert torch.allclose(la, lb, rtol=0, atol=1e-4 * float(la.max() - la.min()))


def test_chain_wait_timeout_sets_status_poisons_and_context_stays_usable():
    # A one-poll limit on the grid-wide waits between chain phases is shorter
    # than the chain's CTAs take to meet: a wait gives up, sets the status bit
    # and the launch runs on; the model is poisoned, the context is not.
    import block_quantized_transformer_gb300 as tq
    w = synth.TINY
    m = build_model(w, device=DEV, max_ctx=64)
    m.set_wait_limit(1)
    tok = torch.tensor([3], dtype=torch.int32, device=DEV)
    for s in range(12):
        p = torch.tensor([s], dtype=torch.int32, device=DEV)
        m.decode_step(tok, p, p)
    with pytest.raises(tq.TqPoisoned, match="device wait timed out"):
        m.status()
    with pytest.raises(tq.TqError, match="closed"):
        m.decode_step(tok, p, p)
    torch.cuda.synchronize()
    run_case(w, w.prompt_len, 4)          # a fresh model on the same device is exact again


def test_decode_chain_alone_matches_the_step():
    # tq_decode_chain enqueues the step's own chain: after a decode step, re-running
    # the last layer's chain over the same activations reproduces the step's head
    import block_quantized_transformer_gb300 as tq
    w = synth.TINY
    m = build_model(w, device=DEV, max_ctx=32)
    prompt = torch.tensor(w.prompt(), dtype=torch.int32, device=DEV)
    m.prefill(prompt)
    with pytest.raises(tq.TqError, match="outside"):
        m.decode_chain(w.n_layers)
    m.decode_chain(0)                       # runs; overwrites the activations
    assert m.status() == 0
    m.close()
