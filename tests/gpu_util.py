"""Helpers of the GPU parity tests (teacher-forced comparison with the oracle)."""
import numpy as np
import torch

import synth
from oracle import model as om


def rel_logit_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| over the oracle's logit range."""
    return float(np.max(np.abs(got - ref)) / (ref.max() - ref.min()))


def top2_margin(ref: np.ndarray) -> float:
    s = np.sort(ref)
    return float(s[-1] - s[-2])


def check_tokens(got_tok, ref_logits, tol):
    """Greedy tokens must equal the oracle's wherever its top-2 margin exceeds
    tol times its logit range; returns the number of steps compared."""
    n = 0
    for t, r in zip(got_tok, ref_logits):
        if top2_margin(r) > tol * (r.max() - r.min()):
            assert t == int(np.argmax(r)), (t, int(np.argmax(r)))
            n += 1
    return n


def gpu_teacher_forced(model, prompt, feed, device):
    """Prefill `prompt`, then one decode step per token of `feed`; returns the
    logits (numpy f64) and greedy tokens of the prefill and of every step."""
    V = model.cfg.vocab
    logits = torch.empty(V, dtype=torch.float32, device=device)
    am = model.prefill(torch.tensor(np.asarray(prompt), dtype=torch.int32, device=device),
                       logits=logits)
    out_l = [logits.double().cpu().numpy()]
    out_t = [int(am.item())]
    P = len(prompt)
    for s, tok in enumerate(feed):
        t = torch.tensor([int(tok)], dtype=torch.int32, device=device)
        p = torch.tensor([P + s], dtype=torch.int32, device=device)
        lg = torch.empty(1, V, dtype=torch.float32, device=device)
        am = model.decode_step(t, p, p.clone(), logits=lg)
        out_l.append(lg[0].double().cpu().numpy())
        out_t.append(int(am.item()))
    return out_l, out_t
