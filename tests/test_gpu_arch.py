"""GPU parity of the sibling layer recipes ("Inferencia local y
arquitecturas", section "El formato"): llama (no per-head Q/K norm), qwen2
(Q/K/V biases) and gemma3-style (tanh-GELU gate, sliding window on a layer
pattern, final logit softcap), each through every path that runs it --
GEMM prefill and GEMV-chain decode over an f32 cache, the flash prefill and
the tensor-core decode attention over an f16 cache, batched decode over a
paged cache -- against the oracle's run of the same recipe, teacher-forced.
Tolerances as in test_gpu_model: 2e-3 of the oracle's logit range with an f32
cache, 1e-2 with f16."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import model as om
from block_quantized_transformer_gb300.synthetic import build_model
from gpu_util import rel_logit_err, check_tokens, gpu_teacher_forced
from test_gpu_batched import _batched_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ARCH = {w.arch: w for w in synth.ARCH_WORKLOADS}


def _run(w, prompt_len, steps, tol):
    prompt = list(w.prompt(n=prompt_len))
    ref = om.OracleModel(w, om.synth_weights(w))
    toks, ref_logits = om.run_greedy(ref, prompt, steps)
    model = build_model(w, device=DEV, max_ctx=prompt_len + steps + 1, max_prefill=prompt_len)
    got_l, got_t = gpu_teacher_forced(model, prompt, toks[:steps], DEV)
    assert model.status() == 0
    model.close()
    errs = [rel_logit_err(g, r) for g, r in zip(got_l, ref_logits)]
    assert max(errs) <= tol, (w.name, max(errs), int(np.argmax(errs)))
    check_tokens(got_t, ref_logits, tol)
    return max(errs)


@pytest.mark.parametrize("arch", ["llama", "qwen2", "gemma3"])
def test_arch_f32_cache(arch):
    err = _run(ARCH[arch], 8, 16, 2e-3)
    print(f"{arch} f32: max rel logit err {err:.2e}")


@pytest.mark.parametrize("arch", ["llama", "qwen2", "gemma3"])
def test_arch_f16_cache_q4_0_long_prompt(arch):
    # 200 prompt tokens: the flash prefill's 64-key tiles, and for gemma3 a
    # 40-key window that starts past the first tiles of later query blocks
    w = dataclasses.replace(ARCH[arch], name=f"{arch}_f16", kv="f16", wtype="q4_0",
                            sliding_window=40 if arch == "gemma3" else 0)
    err = _run(w, 200, 8, 1e-2)
    print(f"{arch} f16 q4_0: max rel logit err {err:.2e}")


@pytest.mark.parametrize("arch", ["qwen2", "gemma3"])
def test_arch_batched_paged(arch):
    w = dataclasses.replace(ARCH[arch], name=f"{arch}_batched", kv="f16", wtype="q4_0")
    _batched_case(w, [5, 17, 9, 30], 8, page_size=32, n_pages=16)


def test_gemma3_window_matters():
    # the same weights with the window off give other logits: the test above
    # is not passing by accident of a window wider than the context
    w = ARCH["gemma3"]
    prompt = list(w.prompt(n=8))
    a = om.OracleModel(w, om.synth_weights(w)).forward_nocache(prompt + [1, 2, 3, 4])
    b = om.OracleModel(dataclasses.replace(w, sliding_window=0), om.synth_weights(w)).forward_nocache(
        prompt + [1, 2, 3, 4])
    assert np.max(np.abs(a - b)) > 1e-3
