"""Host-side bookkeeping of continuous batching (no GPU): row planning with
chunked prefill next to decode rows, page allocation as sequences grow, page
reuse after eviction, and refusal when the pool runs dry."""
from types import SimpleNamespace

import numpy as np
import pytest

from block_quantized_transformer_gb300.batching import PagedBatcher, OutOfPages


def _batcher(n_pages=12, max_batch=4, max_ctx=128, max_prefill=64, chunk=32):
    cfg = SimpleNamespace(page_size=32, max_ctx=max_ctx, max_batch=max_batch, n_pages=n_pages,
                          max_prefill=max_prefill)
    return PagedBatcher(SimpleNamespace(cfg=cfg, device="cpu"), chunk=chunk)


def _live_pages_disjoint(b):
    seen = []
    for s in b.seqs.values():
        seen += s.pages
        assert [int(b.table[s.slot, i]) for i in range(len(s.pages))] == s.pages
    assert len(seen) == len(set(seen))
    assert not (set(seen) & set(b.free))


def test_plan_mixes_prefill_chunks_and_decode_rows():
    b = _batcher()
    a0, a1, a2 = b.admit(range(100, 170)), b.admit(range(5)), b.admit(range(40))
    p = b.plan()
    # slot 0: 32 prompt rows; slot 1: its whole 5-token prompt; slot 2: the 27 rows left in the budget
    assert p.row_seq.tolist() == [0] * 32 + [1] * 5 + [2] * 27
    assert p.row_pos.tolist() == list(range(32)) + list(range(5)) + list(range(27))
    assert p.tokens[:3].tolist() == [100, 101, 102]
    assert p.last_row.tolist() == [31, 36, 63]
    assert p.emits == [False, True, False]
    _live_pages_disjoint(b)
    out = b.commit(p, np.array([7, 8, 9]))
    assert out == {1: 8} and b.seqs[1].next_token == 8
    p = b.plan()
    # slot 0: next chunk at 32..63; slot 1: one decode row at 5; slot 2: the last 13 prompt rows
    assert p.row_seq.tolist() == [0] * 32 + [1] + [2] * 13
    assert p.row_pos.tolist() == list(range(32, 64)) + [5] + list(range(27, 40))
    assert p.tokens[32] == 8
    assert p.emits == [False, True, True]
    assert len(b.seqs[0].pages) == 2 and len(b.seqs[2].pages) == 2
    _live_pages_disjoint(b)


def test_eviction_returns_pages_and_a_new_sequence_reuses_them():
    b = _batcher(n_pages=3, chunk=64)
    s0 = b.admit(range(40))
    s1 = b.admit(range(10))
    b.commit(b.plan(), np.array([1, 2]))
    assert len(b.seqs[s0].pages) == 2 and len(b.seqs[s1].pages) == 1 and b.free_pages() == 0
    pages0 = list(b.seqs[s0].pages)
    b.evict(s0)
    assert b.free_pages() == 2
    s2 = b.admit(range(50))
    assert s2 == s0                                  # the freed slot
    b.commit(b.plan(), np.array([3, 4]))
    assert sorted(b.seqs[s2].pages) == sorted(pages0)  # the evicted sequence's pages, reused
    _live_pages_disjoint(b)


def test_out_of_pages_is_refused():
    b = _batcher(n_pages=2, max_prefill=128, chunk=64)
    b.admit(range(64))
    b.admit(range(10))
    with pytest.raises(OutOfPages):
        b.plan()


def test_admission_limits():
    b = _batcher(max_batch=2)
    b.admit([1])
    b.admit([2])
    with pytest.raises(RuntimeError):
        b.admit([3])
    with pytest.raises(ValueError):
        _batcher().admit([])
