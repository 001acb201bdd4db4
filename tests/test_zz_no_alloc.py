"""The allocation-free greedy head (tq_lm_head_static) against the head that
takes caller scratch (tq_lm_head), through the C ABI.

Some callers of this library cannot allocate device memory -- a plugin inside
a framework that owns the device pool, or a thread that must not risk the
device-wide synchronization of cudaMalloc -- so tq_lm_head_static keeps its
argmax keys in a static device array.  Two calls in a row, with different
inputs, must give what tq_lm_head gives: the array keeps the previous call's
keys, so the second call checks that each call clears what it uses.  This file
is collected last; it passes alone in a fresh process and after the rest."""
import numpy as np
import pytest
import torch

import synth
from oracle import quant
import block_quantized_transformer_gb300 as tq

pytestmark = pytest.mark.gpu


def _head(wtype, vocab, hidden, dev):
    w = synth.host_normal(31, 1, vocab * hidden).reshape(vocab, hidden)
    blocks = torch.from_numpy(quant.quantize(w, wtype)).to(dev)
    return tq.QMat.from_blocks(tq.WTYPES[wtype], blocks, vocab, hidden)


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
def test_static_scratch_head_matches_caller_scratch_head_twice(wtype):
    dev = torch.device("cuda:0")
    vocab, hidden = 30011, 1024
    m = _head(wtype, vocab, hidden, dev)
    gain = torch.from_numpy(synth.host_normal(31, 2, hidden, mean=1.0)).to(dev)
    # the first call's gain is 8x larger, so its logits (and argmax keys) are
    # larger than any of the second call's: keys left over from the first call
    # would win the second call's argmax unless each call clears its rows
    for call, (batch, scale) in enumerate(((7, 8.0), (5, 1.0))):
        x = torch.from_numpy(synth.host_normal(31, 10 + call, batch * hidden, sigma=1.0)
                             .reshape(batch, hidden)).to(dev)
        g = gain * scale
        ref_logits, ref_am = tq.tq_lm_head(m, x, g)
        logits = torch.empty(batch, vocab, dtype=torch.float32, device=dev)
        am = torch.empty(batch, dtype=torch.int32, device=dev)
        got_logits, got_am = tq.tq_lm_head_static(m, x, g, logits=logits, argmax=am)
        torch.cuda.synchronize()
        assert torch.equal(got_am, ref_am), (call, got_am, ref_am)
        # same kernel and inputs: identical logits (the tests' tolerance for this op is 1e-5
        # of the logit range against the oracle; here the two entry points agree exactly)
        assert torch.equal(got_logits, ref_logits)
        assert torch.equal(got_am.long(), got_logits.argmax(dim=1))


def test_static_scratch_head_refuses_oversized_batch():
    dev = torch.device("cuda:0")
    m = _head("q8_0", 64, 256, dev)
    x = torch.zeros(tq.LM_HEAD_STATIC_MAX_BATCH + 1, 256, device=dev)
    gain = torch.ones(256, device=dev)
    with pytest.raises(tq.TqError):
        tq.tq_lm_head_static(m, x, gain)
    import ctypes
    rc = tq.lib().tq_lm_head_static(tq.TQ_Q8_0, m.abi, 64, 256, ctypes.c_void_p(x.data_ptr()),
                                    tq.LM_HEAD_STATIC_MAX_BATCH + 1, ctypes.c_void_p(gain.data_ptr()),
                                    1e-6, None, ctypes.c_void_p(x.data_ptr()), None)
    assert rc == tq.TQ_REFUSED
    assert "TQ_LM_HEAD_STATIC_MAX_BATCH" in tq.tq_last_error()
