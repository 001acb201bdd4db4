"""Temperature / top-p sampling of one row of logits (oracle; test infrastructure).

Restates the sampler of "Всередині LLM: чисте виконання на Python для
Qwen3-0.6B на MLX", step 8 (``sample(logits, temperature, top_p)``), in float64:

* temperature 0: greedy, the index of the largest logit;
* otherwise the logits are divided by the temperature and turned into
  probabilities with a softmax;
* top-p: the tokens are ordered by descending probability and the smallest
  prefix whose cumulative probability reaches top_p is kept (the count of
  prefix sums below top_p, plus one); the kept probabilities are renormalised;
* one token is drawn from the kept set.

Readings where the page leaves a step open:

* equal probabilities are ordered by ascending token index (a stable sort);
* the draw is an inverse-CDF pick with a uniform number u in [0, 1) supplied
  by the caller: the first kept token, in the same order, whose cumulative
  renormalised probability exceeds u (the page draws with its library's
  categorical sampler, whose use of the random bits it does not fix);
* argmax ties go to the lowest index.
"""
from __future__ import annotations

import numpy as np


def nucleus(logits: np.ndarray, temperature: float, top_p: float):
    """(order, kept probabilities renormalised): the kept tokens in descending
    order of probability and their renormalised probabilities."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max()
    p = np.exp(z)
    p = p / p.sum()
    order = np.argsort(-p, kind="stable")          # ties: ascending index
    sp = p[order]
    cum = np.cumsum(sp)
    cutoff = int(np.sum(cum < top_p)) + 1
    cutoff = min(cutoff, len(sp))
    kept = sp[:cutoff]
    return order[:cutoff], kept / kept.sum()


def sample(logits: np.ndarray, temperature: float, top_p: float, u: float) -> int:
    """The token drawn for the uniform number u in [0, 1)."""
    if temperature == 0:
        return int(np.argmax(logits))
    order, q = nucleus(logits, temperature, top_p)
    cum = np.cumsum(q)
    i = int(np.sum(cum <= u))                       # first with cum > u
    return int(order[min(i, len(order) - 1)])


def boundary_distance(logits: np.ndarray, temperature: float, top_p: float, u: float) -> float:
    """How far u and top_p sit from the decisions they make (the smallest gap
    between u and a kept token's cumulative probability, and between top_p and
    the cumulative probability at the cutoff); a test uses it to keep only
    draws that a few ulps of rounding cannot flip."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max()
    p = np.exp(z)
    p = p / p.sum()
    sp = p[np.argsort(-p, kind="stable")]
    cum = np.cumsum(sp)
    c = int(np.sum(cum < top_p))
    gap_p = min(abs(top_p - cum[c]) if c < len(cum) else 1.0, abs(top_p - cum[c - 1]) if c > 0 else 1.0)
    kept = sp[:min(c + 1, len(sp))]
    qc = np.cumsum(kept / kept.sum())
    gap_u = float(np.min(np.abs(qc - u)))
    return min(gap_p, gap_u)
