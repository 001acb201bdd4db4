"""The seeded input generator: pinned to Philox4x32-10's published
known-answer vectors; the NumPy, C and (on a GPU) CUDA versions agree bit for bit."""
import numpy as np
import pytest

import synth
from conftest import golden


def _kat():
    rows = []
    for line in open(__import__("os").path.join(synth._HERE, "..", "tests", "golden",
                                                 "philox4x32_10_kat.txt")):
        if line.strip() and not line.startswith("#"):
            rows.append([int(t, 16) for t in line.split()])
    return rows


def test_philox_known_answers_numpy():
    for r in _kat():
        out = synth.philox4x32_10(([r[0]], [r[1]], [r[2]], [r[3]]), (r[4], r[5]))
        assert [int(o[0]) for o in out] == r[6:10]


def test_philox_known_answers_c():
    for r in _kat():
        assert [int(v) for v in synth.host_philox(r[0:4], (r[4], r[5]))] == r[6:10]


def test_host_matches_numpy_bitwise():
    a = synth.normal(11, 3, 50_000, first=7_000_000_000)
    b = synth.host_normal(11, 3, 50_000, first=7_000_000_000)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    g1 = synth.normal(11, 4, 1000, mean=1.0)
    g2 = synth.host_normal(11, 4, 1000, mean=1.0)
    assert np.array_equal(g1.view(np.uint32), g2.view(np.uint32))
    t1 = synth.uniform_below(2, 9, 10_000, 151936)
    t2 = synth.host_uniform_below(2, 9, 10_000, 151936)
    assert np.array_equal(t1, t2) and t1.min() >= 0 and t1.max() < 151936


def test_normal_moments():
    v = synth.host_normal(1, 1, 2_000_000).astype(np.float64)
    assert abs(v.mean()) < 1e-4
    assert abs(v.std() - 0.02) < 1e-4
    # Irwin-Hall(8) support is +-4.9 sigma
    assert np.abs(v).max() <= 4.9 * 0.02 + 1e-6


def test_workload_streams_distinct():
    w = synth.TINY
    names = w.matrices() + w.gains()
    streams = [w.stream_of(n) for n in names]
    assert len(set(streams)) == len(streams)
    assert w.weight_count() == sum(int(np.prod(w.matrix_shape(n))) for n in w.matrices())


def test_row_slices_match_full_tensor():
    w = synth.TINY
    full = synth.host_tensor(w, "blk.1.ffn_down")
    part = synth.host_tensor(w, "blk.1.ffn_down", rows=slice(10, 20))
    assert np.array_equal(full[10:20], part)


def test_context_lengths_in_range():
    w = synth.QWEN3_8B_Q4_BATCHED
    L = w.context_lengths()
    assert L.shape == (32,) and L.min() >= 512 and L.max() <= 8192
