"""GPU parity of continuous batching: several sequences admitted at different
steps, their prompts prefilled in chunks inside the same tq_step calls as
other sequences' decode tokens, one evicted mid-way and its pages reused by a
newly admitted sequence; every emitted logit row is compared with the
oracle's run of that sequence alone, teacher-forced on the oracle's greedy
tokens.  Tolerance: 2e-3 of the oracle's logit range with an f32 cache, 1e-2
with f16."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import model as om
from block_quantized_transformer_gb300.batching import PagedBatcher
from block_quantized_transformer_gb300.synthetic import build_model
from gpu_util import rel_logit_err, check_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _scenario(w, tol):
    prompts = {"A": list(w.prompt(0, n=45)), "B": list(w.prompt(1, n=6)), "C": list(w.prompt(2, n=21)),
               "D": list(w.prompt(3, n=9))}
    ref = om.OracleModel(w, om.synth_weights(w))
    oracle = {k: om.run_greedy(ref, p, 16) for k, p in prompts.items()}   # (tokens, logits)
    # four pages: B's single page is the only free one when D arrives, so D reuses it
    model = build_model(w, device=DEV, max_batch=4, max_ctx=96, max_prefill=48, page_size=32, n_pages=4)
    b = PagedBatcher(model, chunk=16)
    slot = {"A": b.admit(prompts["A"]), "B": b.admit(prompts["B"])}
    name = {v: k for k, v in slot.items()}
    got = {k: [] for k in prompts}
    got_tok = {k: [] for k in prompts}
    logits = torch.empty(4, w.vocab, device=DEV)
    for step in range(14):
        if step == 2:
            slot["C"] = b.admit(prompts["C"])
            name[slot["C"]] = "C"
        if step == 5:                                  # B finishes; D takes its slot and pages
            freed = list(b.seqs[slot["B"]].pages)
            b.evict(slot["B"])
            del name[slot["B"]]
            slot["D"] = b.admit(prompts["D"])
            name[slot["D"]] = "D"
        if step == 6:
            assert b.seqs[slot["D"]].pages == freed
        emitted = b.step(logits=logits)
        lg = logits.double().cpu().numpy()
        for k, s in enumerate(b.last_plan.slots):
            if s not in emitted:
                continue
            seq = name[s]
            i = len(got[seq])
            got[seq].append(lg[k])
            got_tok[seq].append(emitted[s])
            # teacher forcing: the next decode step feeds the oracle's token
            b.seqs[s].next_token = int(oracle[seq][0][i])
    assert model.status() == 0
    model.close()
    worst = 0.0
    for seq, rows in got.items():
        assert len(rows) >= 3, (seq, len(rows))
        ref_l = oracle[seq][1][:len(rows)]
        errs = [rel_logit_err(g, r) for g, r in zip(rows, ref_l)]
        worst = max(worst, max(errs))
        assert max(errs) <= tol, (seq, max(errs), int(np.argmax(errs)))
        check_tokens(got_tok[seq], ref_l, tol)
    return worst


def test_continuous_batching_f16_cache():
    w = dataclasses.replace(synth.TINY, name="tiny_batching_f16", kv="f16", wtype="q4_0")
    worst = _scenario(w, 1e-2)
    print(f"continuous batching f16: max rel logit err {worst:.3e}")


def test_continuous_batching_f32_cache():
    w = dataclasses.replace(synth.TINY, name="tiny_batching_f32")
    worst = _scenario(w, 2e-3)
    print(f"continuous batching f32: max rel logit err {worst:.3e}")


@pytest.mark.parametrize("kv", ["f16", "f32"])
def test_bad_sequence_index_sets_status_and_poisons(kv):
    """A row whose sequence index lies outside [0, max_batch) touches no
    cache row of another sequence and nothing out of bounds: its K/V are not
    appended, its attention reads stay inside the cache, and the step sets the
    out-of-range status bit, which poisons the model."""
    import block_quantized_transformer_gb300 as tq
    w = dataclasses.replace(synth.TINY, kv=kv)
    model = build_model(w, device=DEV, max_batch=2, max_ctx=64, max_prefill=48, page_size=32, n_pages=4)
    n = 34
    tok = torch.ones(n, dtype=torch.int32, device=DEV)
    seq = torch.zeros(n, dtype=torch.int32, device=DEV)
    seq[-1] = 7
    pos = torch.arange(n, dtype=torch.int32, device=DEV)
    pos[-1] = 0
    last = torch.tensor([n - 2, n - 1], dtype=torch.int32, device=DEV)
    bt = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device=DEV)
    model.step(tok, seq, pos, last, block_table=bt)
    with pytest.raises(tq.TqPoisoned, match="out of range"):
        model.status()


@pytest.mark.parametrize("base,kv", [(synth.TINY, "f16"), (synth.TINY, "f32"), (synth.TINY_GEMMA3, "f16")])
def test_mixed_step_flash_blocks_tiny(base, kv):
    """head_dim 64, two query heads per KV head (flash blocks of 64 rows): one
    step carries a 70-row prompt of sequence 0 (rows 0..63 one flash block,
    rows 64..69 with sequence 1's 5-row prompt left to the row-wise kernel),
    then both sequences decode; pages in a shuffled order; the gemma3-style
    recipe puts the sliding window on alternate layers."""
    w = dataclasses.replace(base, kv=kv)
    tol = 2e-3 if kv == "f32" else 1e-2
    ref = om.OracleModel(w, om.synth_weights(w))
    pa, pb = list(w.prompt(0, n=70)), list(w.prompt(1, n=5))
    ca, cb = ref.new_cache(), ref.new_cache()
    ref_l = [[ref.forward(pa, ca, 0)], [ref.forward(pb, cb, 0)]]
    nxt = [om.argmax(ref_l[0][0]), om.argmax(ref_l[1][0])]
    ref_l[0].append(ref.forward([nxt[0]], ca, 70))
    ref_l[1].append(ref.forward([nxt[1]], cb, 5))

    model = build_model(w, device=DEV, max_batch=2, max_ctx=128, max_prefill=80, page_size=32, n_pages=8)
    bt = torch.tensor([[5, 2, 7, 0], [3, 6, 1, 4]], dtype=torch.int32, device=DEV)
    i32 = lambda v: torch.tensor(v, dtype=torch.int32, device=DEV)
    steps = [(pa + pb, [0] * 70 + [1] * 5, list(range(70)) + list(range(5)), [69, 74]),
             (nxt, [0, 1], [70, 5], [0, 1])]
    got_l, got_t = [[], []], [[], []]
    for tok, seq, pos, last in steps:
        lg = torch.empty(2, w.vocab, dtype=torch.float32, device=DEV)
        am = model.step(i32(tok), i32(seq), i32(pos), i32(last), block_table=bt, logits=lg)
        lg_h, am_h = lg.double().cpu().numpy(), am.cpu().numpy()
        for b in range(2):
            got_l[b].append(lg_h[b])
            got_t[b].append(int(am_h[b]))
    assert model.status() == 0
    model.close()
    for b in range(2):
        errs = [rel_logit_err(g, r) for g, r in zip(got_l[b], ref_l[b])]
        assert max(errs) <= tol, (b, errs)
        check_tokens(got_t[b], ref_l[b], tol)
