"""Continuous batching over a paged KV cache (host-side bookkeeping only).

Sequences are admitted with a prompt, prefilled in chunks in the same steps
as other sequences' decode tokens, and evicted when done; every step is one
``tq_step`` call over the rows of all sequences that have work.  A sequence's
cache is the list of pages in its block-table row: pages are taken from a
free pool as the sequence grows and returned to it on eviction, so a new
sequence reuses them (it writes its own K/V from position 0 before reading).

This module decides which rows go into a step; the forward pass itself runs
in the library's kernels.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch


class OutOfPages(RuntimeError):
    """The pool has no free page for a sequence that must grow."""


@dataclass
class Sequence:
    slot: int
    prompt: List[int]
    consumed: int = 0                 # prompt tokens already in the cache
    length: int = 0                   # tokens in the cache
    pages: List[int] = field(default_factory=list)
    next_token: Optional[int] = None  # the token to feed at the next decode step
    outputs: List[int] = field(default_factory=list)

    @property
    def prefilling(self) -> bool:
        return self.consumed < len(self.prompt)


@dataclass
class StepPlan:
    tokens: np.ndarray      # [n_rows] int32
    row_seq: np.ndarray     # [n_rows] block-table row of each token
    row_pos: np.ndarray     # [n_rows] position / cache index
    last_row: np.ndarray    # [n_seq] row whose logits each sequence gets
    slots: List[int]        # the sequences of the step, in last_row order
    emits: List[bool]       # whether that sequence's row yields its next token


class PagedBatcher:
    """Admission, chunked prefill, decode and eviction for one model.

    ``model`` needs a paged cache (page_size > 0); ``chunk`` caps the prompt
    rows a sequence contributes to one step, ``max_rows`` the rows of a step
    (at most the model's max_prefill)."""

    def __init__(self, model, chunk: int = 64, max_rows: Optional[int] = None):
        cfg = model.cfg
        if cfg.page_size <= 0:
            raise ValueError("continuous batching needs a paged cache (page_size > 0)")
        self.model = model
        self.page_size = cfg.page_size
        self.pages_per_seq = cfg.max_ctx // cfg.page_size
        self.max_seqs = cfg.max_batch
        self.chunk = int(chunk)
        self.max_rows = int(max_rows or cfg.max_prefill)
        if self.max_rows > cfg.max_prefill:
            raise ValueError("max_rows exceeds the model's max_prefill")
        self.free = deque(range(cfg.n_pages))
        self.seqs: Dict[int, Sequence] = {}
        self.table = np.full((self.max_seqs, self.pages_per_seq), 0, dtype=np.int32)

    # -- admission / eviction
    def admit(self, prompt) -> int:
        """Admit a sequence; returns its slot (block-table row)."""
        prompt = [int(t) for t in prompt]
        if not prompt:
            raise ValueError("empty prompt")
        if len(prompt) > self.pages_per_seq * self.page_size:
            raise ValueError("prompt longer than max_ctx")
        free_slots = [s for s in range(self.max_seqs) if s not in self.seqs]
        if not free_slots:
            raise RuntimeError("no free sequence slot")
        slot = free_slots[0]
        self.seqs[slot] = Sequence(slot=slot, prompt=prompt)
        return slot

    def evict(self, slot: int) -> Sequence:
        """Remove a sequence and return its pages to the pool."""
        seq = self.seqs.pop(slot)
        self.free.extend(seq.pages)
        seq.pages = []
        return seq

    def free_pages(self) -> int:
        return len(self.free)

    # -- planning
    def _grow(self, seq: Sequence, new_len: int):
        need = (new_len + self.page_size - 1) // self.page_size
        while len(seq.pages) < need:
            if not self.free:
                raise OutOfPages(f"no free page for slot {seq.slot}")
            p = self.free.popleft()
            self.table[seq.slot, len(seq.pages)] = p
            seq.pages.append(p)

    def plan(self) -> Optional[StepPlan]:
        """Rows of the next step: a prompt chunk of every prefilling sequence
        and the next token of every decoding one, in slot order, within the
        row budget.  Pages for the new positions are taken here."""
        toks, rseq, rpos, last, slots, emits = [], [], [], [], [], []
        for slot in sorted(self.seqs):
            seq = self.seqs[slot]
            if seq.prefilling:
                n = min(self.chunk, len(seq.prompt) - seq.consumed, self.max_rows - len(toks))
                if n <= 0:
                    continue
                feed = seq.prompt[seq.consumed:seq.consumed + n]
            elif seq.next_token is not None:
                if len(toks) + 1 > self.max_rows:
                    continue
                feed = [seq.next_token]
            else:
                continue
            if seq.length + len(feed) > self.pages_per_seq * self.page_size:
                continue                    # full: the caller should evict it
            self._grow(seq, seq.length + len(feed))
            for k, t in enumerate(feed):
                toks.append(t)
                rseq.append(slot)
                rpos.append(seq.length + k)
            last.append(len(toks) - 1)
            slots.append(slot)
            emits.append(not seq.prefilling or seq.consumed + len(feed) == len(seq.prompt))
        if not toks:
            return None
        return StepPlan(np.asarray(toks, np.int32), np.asarray(rseq, np.int32), np.asarray(rpos, np.int32),
                        np.asarray(last, np.int32), slots, emits)

    def commit(self, plan: StepPlan, out_tokens) -> Dict[int, int]:
        """Advance the sequences of a planned step by its results: lengths,
        consumed prompt, and the next token of every sequence that emitted one
        (returned as {slot: token})."""
        emitted = {}
        counts = np.bincount(plan.row_seq, minlength=self.max_seqs)
        for k, slot in enumerate(plan.slots):
            seq = self.seqs[slot]
            n = int(counts[slot])
            if seq.prefilling:
                seq.consumed += n
            seq.length += n
            if plan.emits[k]:
                tok = int(out_tokens[k])
                seq.next_token = tok
                seq.outputs.append(tok)
                emitted[slot] = tok
        return emitted

    # -- one step on the device
    def step(self, logits: Optional[torch.Tensor] = None) -> Dict[int, int]:
        """Plan, run one tq_step, commit; returns the emitted greedy tokens.
        `logits` (optional, [max_seqs][vocab]) receives each stepped
        sequence's logits in the plan's order."""
        plan = self.plan()
        if plan is None:
            return {}
        self.last_plan = plan
        dev = self.model.device
        out = self.model.step(torch.from_numpy(plan.tokens).to(dev), torch.from_numpy(plan.row_seq).to(dev),
                              torch.from_numpy(plan.row_pos).to(dev), torch.from_numpy(plan.last_row).to(dev),
                              block_table=torch.from_numpy(self.table).to(dev),
                              logits=None if logits is None else logits[:len(plan.slots)])
        return self.commit(plan, out.cpu().numpy())
