"""Host-side checks of the C ABI and its binding (no GPU work): the library
loads, exports every entry point include/tq.h declares, validates
configurations on the host, and the binding range-checks integers and keeps
handle discipline."""
import copy
import ctypes
import os
import pickle
import re

import pytest

import block_quantized_transformer_gb300 as tq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_entry_points():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    return sorted(set(re.findall(r"TQ_API [^;(]*?\b(tq_\w+)\(", src)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(tq.LIB_PATH):
        from block_quantized_transformer_gb300 import build
        build.build()


def test_exports_every_declared_entry_point():
    declared = header_entry_points()
    assert len(declared) >= 16
    L = tq.lib()
    missing = [n for n in declared if not hasattr(L, n)]
    assert not missing, missing
    assert sorted(tq.EXPORTS) == declared


def _cfg(**kw):
    base = dict(vocab=4096, hidden=256, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64,
                ffn=768, rms_eps=1e-6, rope_theta=1e6, wtype=tq.TQ_Q8_0, kvtype=tq.TQ_KV_F32,
                max_batch=1, max_ctx=64, max_prefill=16, page_size=0, n_pages=0)
    base.update(kw)
    return tq.TqConfig(**base)


def test_workspace_and_cache_sizes():
    c = _cfg()
    ws = tq.tq_workspace_bytes(c)
    assert ws > 0 and ws % 256 == 0
    assert tq.tq_kv_cache_bytes(c) == 2 * 1 * 2 * 64 * 64 * 4
    c16 = _cfg(kvtype=tq.TQ_KV_F16)
    assert tq.tq_kv_cache_bytes(c16) == 2 * 1 * 2 * 64 * 64 * 2
    paged = _cfg(page_size=32, n_pages=10, max_ctx=64)
    assert tq.tq_kv_cache_bytes(paged) == 2 * 10 * 2 * 32 * 64 * 4


@pytest.mark.parametrize("bad,msg", [
    (dict(head_dim=96), "head_dim"),
    (dict(n_heads=6, n_kv_heads=4), "multiple"),
    (dict(n_heads=48, n_kv_heads=3), "1, 2, 4 or 8"),
    (dict(wtype=3), "wtype"),
    (dict(kvtype=7), "kvtype"),
    (dict(hidden=100), "GEMV"),
    (dict(max_batch=0), "max_batch"),
    (dict(page_size=48, n_pages=4), "page_size"),
    (dict(page_size=32, n_pages=4, max_ctx=40), "multiple of page_size"),
    (dict(page_size=32, n_pages=0), "n_pages"),
    (dict(arch=4), "arch"),
    (dict(arch=-1), "arch"),
    (dict(arch=1, sliding_window=8), "gemma3"),
    (dict(arch=0, logit_softcap=30.0), "gemma3"),
    (dict(arch=3, sliding_window=-2), ">= 0"),
    (dict(arch=3, logit_softcap=-1.0), ">= 0"),
])
def test_invalid_configs_refused_with_reason(bad, msg):
    assert tq.tq_workspace_bytes(_cfg(**bad)) == 0
    assert msg in tq.tq_last_error()


def test_null_arguments_refused_without_gpu():
    L = tq.lib()
    assert L.tq_model_create(None, None, None, None, None, None) == tq.TQ_REFUSED
    h = ctypes.c_void_p()
    assert L.tq_model_create(ctypes.byref(_cfg()), None, None, None, None, ctypes.byref(h)) == tq.TQ_REFUSED
    assert L.tq_prefill(None, 0, None, 1, 0, None, None, None, None) == tq.TQ_REFUSED
    assert "NULL" in tq.tq_last_error()
    assert L.tq_decode_step(None, 1, None, None, None, None, None, None, None) == tq.TQ_REFUSED
    assert L.tq_model_poisoned(None) == 0
    L.tq_model_free(None)                               # ignored
    assert L.tq_repack(5, None, 1, 32, None, None, None) == tq.TQ_REFUSED
    assert L.tq_quantize(2, None, 1, 33, None, None) == tq.TQ_REFUSED
    assert L.tq_repack(2, None, 0, 256, None, None, None) == tq.TQ_OK  # empty is a no-op
    assert L.tq_repack(2, None, 1, 32, None, None, None) == tq.TQ_REFUSED  # tiles need cols % 256 == 0


def test_tiled_matrix_sizes():
    """Rows pad to a multiple of 16; 16 (Q4_0) or 32 (Q8_0) code bytes and one
    fp16 scale per block."""
    assert tq.tq_qmat_bytes(tq.TQ_Q4_0, 16, 256) == (16 * 8 * 16, 16 * 8 * 2)
    assert tq.tq_qmat_bytes(tq.TQ_Q4_0, 17, 512) == (32 * 16 * 16, 32 * 16 * 2)
    assert tq.tq_qmat_bytes(tq.TQ_Q8_0, 151936, 4096) == (151936 * 128 * 32, 151936 * 128 * 2)
    assert tq.tq_qmat_bytes(tq.TQ_Q8_0, 0, 256) == (0, 0)
    with pytest.raises(tq.TqError):
        tq.tq_qmat_bytes(tq.TQ_Q4_0, 16, 288)


def test_binding_range_checks_before_the_library():
    with pytest.raises(tq.TqError, match="must be an int"):
        tq._int("n", 1.5, 0, 10)
    with pytest.raises(tq.TqError, match="must be an int"):
        tq._int("n", True, 0, 10)
    with pytest.raises(tq.TqError, match="outside"):
        tq._int("n", 2**31, *tq.I32)
    with pytest.raises(tq.TqError, match="outside"):
        tq._int("n", -1, 0, 10)


def test_model_handle_discipline_without_gpu():
    m = tq.Model.__new__(tq.Model)
    m._handle = None
    import threading
    m._thread = threading.get_ident()
    with pytest.raises(TypeError):
        copy.copy(m)
    with pytest.raises(TypeError):
        copy.deepcopy(m)
    with pytest.raises(TypeError):
        pickle.dumps(m)
    with pytest.raises(tq.TqError, match="closed"):
        m._h()
    m.close()
    m.close()                                           # idempotent


def test_gemm_scratch_bytes():
    """fp16 activation rows (2 B per row and input), one output scale per
    row, split-K partial sums (16 splits, at most 4M floats) and 4096 split
    counters, each 256-byte aligned; 0 for shapes the GEMM does not take."""
    L = tq.lib()
    up = lambda n: (n + 255) // 256 * 256
    for rows, n_rows, cols in [(16, 1, 256), (4096, 32, 4096), (24576, 2048, 12288), (77, 7, 768)]:
        part = min(16 * n_rows * rows, 4 << 20)
        want = up(n_rows * cols * 2) + up(n_rows * 4) + up(part * 4) + up(4096 * 4)
        assert L.tq_gemm_scratch_bytes(rows, n_rows, cols) == want
    for rows, n_rows, cols in [(16, 0, 256), (16, 4, 0), (16, 4, 288), (16, 4, 12544), (0, 4, 256)]:
        assert L.tq_gemm_scratch_bytes(rows, n_rows, cols) == 0


def test_layer_recipes_accepted_and_qwen2_holds_its_biases():
    base = tq.tq_workspace_bytes(_cfg())
    assert tq.tq_workspace_bytes(_cfg(arch=1)) == base
    assert tq.tq_workspace_bytes(_cfg(arch=3, sliding_window=512, sliding_pattern=6, logit_softcap=30.0)) == base
    q2 = tq.tq_workspace_bytes(_cfg(arch=2))
    # the q, k and v biases of both layers side by side: 2 * (4 + 2 * 2) * 64 floats
    assert q2 - base == (2 * (4 + 2 * 2) * 64 * 4 + 255) // 256 * 256
