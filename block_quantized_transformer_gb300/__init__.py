"""Python binding of libtq.so: block-quantized (Q8_0 / Q4_0) Qwen3-style decode
on one GB300.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels behind the C ABI (include/tq.h); PyTorch provides device memory and
streams.  The functions named ``tq_*`` mirror the C entry points one for one;
``Model``, ``QMat`` and the small helpers wrap them.

Conventions follow the tessl_torch README ("Handle ownership, closing and
errors"): a handle is freed exactly once (``Model.close()``, idempotent; copies
and pickling are refused); a handle is used from the thread that made it;
every integer headed for a C field is range-checked first; a refusal (status
1) raises ``TqError`` and leaves the model usable; a library failure (status 2)
raises ``TqPoisoned`` and the model refuses further work.  There is no CPU
fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("TQ_LIB", os.path.join(_PKG, "_build", "libtq.so"))

TQ_OK, TQ_REFUSED, TQ_INTERNAL = 0, 1, 2
TQ_Q4_0, TQ_AFFINE4, TQ_Q8_0 = 2, 4, 8
TQ_KV_F32, TQ_KV_F16 = 0, 1
TQ_DEV_BAD_TOKEN, TQ_DEV_KV_OVERFLOW, TQ_DEV_WAIT_TIMEOUT = 1, 2, 4
WTYPES = {"q4_0": TQ_Q4_0, "q8_0": TQ_Q8_0, "affine4": TQ_AFFINE4}
BLOCK_BYTES = {TQ_Q4_0: 18, TQ_Q8_0: 34}
QS_BYTES = {TQ_Q4_0: 16, TQ_Q8_0: 32, TQ_AFFINE4: 16}  # code bytes per 32 inputs in the tiled layout

EXPORTS = ("tq_workspace_bytes", "tq_kv_cache_bytes", "tq_model_create", "tq_prefill",
           "tq_decode_step", "tq_step", "tq_decode_step_graph", "tq_decode_chain", "tq_model_status",
           "tq_model_set_wait_limit",
           "tq_model_poisoned",
           "tq_decode_launches", "tq_model_free", "tq_last_error", "tq_qmat_bytes", "tq_repack", "tq_quantize",
           "tq_dequantize", "tq_gemv", "tq_gemm_scratch_bytes", "tq_gemm", "tq_swiglu_gemv", "tq_lm_head",
           "tq_sample", "tq_lm_head_static", "tq_quantize_affine4", "tq_repack_affine4")
LM_HEAD_STATIC_MAX_BATCH = 4096


class TqError(RuntimeError):
    """The library refused a call (bad argument); nothing was enqueued."""


class TqPoisoned(TqError):
    """A CUDA error or device status bit: the model is closed for further work."""


# ----------------------------------------------------------------------------- ABI structs

class TqConfig(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("wtype", ctypes.c_int32),
                ("kvtype", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32), ("max_prefill", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("n_pages", ctypes.c_int32),
                ("arch", ctypes.c_int32), ("sliding_window", ctypes.c_int32),
                ("sliding_pattern", ctypes.c_int32), ("logit_softcap", ctypes.c_float)]


class TqQmat(ctypes.Structure):
    _fields_ = [("qs_dev", ctypes.c_void_p), ("d_dev", ctypes.c_void_p)]


class TqLayer(ctypes.Structure):
    _fields_ = [(n, TqQmat) for n in ("attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate",
                                      "ffn_up", "ffn_down")] + \
               [(n, ctypes.c_void_p) for n in ("attn_norm_dev", "ffn_norm_dev",
                                               "attn_q_norm_dev", "attn_k_norm_dev",
                                               "attn_q_bias_dev", "attn_k_bias_dev",
                                               "attn_v_bias_dev")]


class TqWeights(ctypes.Structure):
    _fields_ = [("token_embd", TqQmat), ("output", TqQmat), ("output_norm_dev", ctypes.c_void_p),
                ("layers", ctypes.POINTER(TqLayer))]


_lib = None
_lib_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load libtq.so (raises if it has not been built: there is no fallback)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise TqError(f"libtq.so not built at {LIB_PATH}; run "
                              "block_quantized_transformer_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            cfgp = ctypes.POINTER(TqConfig)
            sig = {
                "tq_workspace_bytes": (ctypes.c_size_t, [cfgp]),
                "tq_kv_cache_bytes": (ctypes.c_size_t, [cfgp]),
                "tq_model_create": (i32, [cfgp, ctypes.POINTER(TqWeights), vp, vp, vp,
                                          ctypes.POINTER(vp)]),
                "tq_prefill": (i32, [vp, i32, vp, i32, i32, vp, vp, vp, vp]),
                "tq_decode_step": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, vp]),
                "tq_decode_step_graph": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, vp]),
                "tq_step": (i32, [vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp]),
                "tq_model_status": (i32, [vp, vp, ctypes.POINTER(ctypes.c_uint32)]),
                "tq_model_set_wait_limit": (i32, [vp, ctypes.c_uint32]),
                "tq_decode_chain": (i32, [vp, i32, vp]),
                "tq_model_poisoned": (ctypes.c_int, [vp]),
                "tq_decode_launches": (i32, [vp, i32]),
                "tq_model_free": (None, [vp]),
                "tq_last_error": (ctypes.c_char_p, []),
                "tq_qmat_bytes": (i32, [i32, i64, i64, ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64)]),
                "tq_repack": (i32, [i32, vp, i64, i64, vp, vp, vp]),
                "tq_quantize": (i32, [i32, vp, i64, i64, vp, vp]),
                "tq_dequantize": (i32, [i32, TqQmat, i64, i64, i64, vp, vp]),
                "tq_gemv": (i32, [i32, TqQmat, i32, i32, vp, i32, vp, vp, vp]),
                "tq_gemm_scratch_bytes": (ctypes.c_size_t, [i32, i32, i32]),
                "tq_gemm": (i32, [i32, TqQmat, i32, i32, vp, i32, vp, vp, vp, vp]),
                "tq_swiglu_gemv": (i32, [i32, TqQmat, TqQmat, i32, i32, vp, i32, vp, f32, vp, vp]),
                "tq_lm_head": (i32, [i32, TqQmat, i32, i32, vp, i32, vp, f32, vp, vp, vp, vp]),
                "tq_lm_head_static": (i32, [i32, TqQmat, i32, i32, vp, i32, vp, f32, vp, vp, vp]),
                "tq_sample": (i32, [vp, i32, i32, vp, vp, vp, vp, vp]),
                "tq_quantize_affine4": (i32, [vp, i64, i64, vp, vp, vp, vp]),
                "tq_repack_affine4": (i32, [vp, vp, vp, i64, i64, vp, vp, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def exported_symbols() -> list:
    L = lib()
    return [n for n in EXPORTS if hasattr(L, n)]


# ----------------------------------------------------------------------------- checks

def _int(name: str, v, lo: int, hi: int) -> int:
    if isinstance(v, bool) or not isinstance(v, int):
        raise TqError(f"{name} must be an int (got {type(v).__name__})")
    if not lo <= v <= hi:
        raise TqError(f"{name}={v} outside [{lo}, {hi}]")
    return v


I32 = (-2**31, 2**31 - 1)
I64 = (-2**63, 2**63 - 1)


def _dev(t: Optional[torch.Tensor], name: str, dtype=None, min_numel: int = 0):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TqError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library works on the current device: another GPU's memory would fault
        raise TqError(f"{name} is on {t.device}, but the current device is "
                      f"cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise TqError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TqError(f"{name} must have dtype {dtype} (got {t.dtype})")
    if t.numel() < min_numel:
        raise TqError(f"{name} holds {t.numel()} elements, needs {min_numel}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device=None) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _status(rc: int, what: str):
    if rc == TQ_OK:
        return
    msg = lib().tq_last_error().decode(errors="replace")
    if rc == TQ_REFUSED:
        raise TqError(f"{what}: {msg}")
    raise TqPoisoned(f"{what}: {msg}")


# ----------------------------------------------------------------------------- raw entry points

def tq_workspace_bytes(cfg: TqConfig) -> int:
    return int(lib().tq_workspace_bytes(ctypes.byref(cfg)))


def tq_kv_cache_bytes(cfg: TqConfig) -> int:
    return int(lib().tq_kv_cache_bytes(ctypes.byref(cfg)))


def tq_last_error() -> str:
    return lib().tq_last_error().decode(errors="replace")


def tq_qmat_bytes(wtype: int, rows: int, cols: int) -> tuple:
    """(qs bytes, d bytes) of a [rows][cols] matrix in the tiled layout."""
    _int("rows", rows, 0, I64[1])
    _int("cols", cols, 0, I64[1])
    q, d = ctypes.c_int64(0), ctypes.c_int64(0)
    _status(lib().tq_qmat_bytes(wtype, rows, cols, ctypes.byref(q), ctypes.byref(d)), "tq_qmat_bytes")
    return q.value, d.value


def tq_repack(wtype: int, blocks: torch.Tensor, rows: int, cols: int, qs: torch.Tensor,
              d: torch.Tensor) -> None:
    """GGUF-order blocks -> tiled layout; qs/d hold the rows padded to a multiple of 16."""
    _int("rows", rows, 0, I64[1])
    _int("cols", cols, 0, I64[1])
    nb = cols // 32
    qb, db = tq_qmat_bytes(wtype, rows, cols)
    rc = lib().tq_repack(wtype, _dev(blocks, "blocks", torch.uint8, rows * nb * BLOCK_BYTES[wtype]),
                         rows, cols, _dev(qs, "qs", torch.uint8, qb),
                         _dev(d, "d", torch.int16, db // 2), _stream())
    _status(rc, "tq_repack")


def tq_quantize(wtype: int, w: torch.Tensor, rows: int, cols: int, blocks: torch.Tensor) -> None:
    _int("rows", rows, 0, I64[1])
    _int("cols", cols, 0, I64[1])
    rc = lib().tq_quantize(wtype, _dev(w, "w", torch.float32, rows * cols), rows, cols,
                           _dev(blocks, "blocks", torch.uint8, rows * (cols // 32) * BLOCK_BYTES[wtype]),
                           _stream())
    _status(rc, "tq_quantize")


def tq_quantize_affine4(w: torch.Tensor, rows: int, cols: int, words: torch.Tensor, scales: torch.Tensor,
                        biases: torch.Tensor) -> None:
    """f32 [rows][cols] -> MLX-layout affine 4-bit groups: words int32 [rows][cols/8],
    scales and biases int16 (bf16 bit patterns) [rows][cols/64]."""
    _int("rows", rows, 0, I64[1])
    _int("cols", cols, 0, I64[1])
    rc = lib().tq_quantize_affine4(_dev(w, "w", torch.float32, rows * cols), rows, cols,
                                   _dev(words, "words", torch.int32, rows * (cols // 8)),
                                   _dev(scales, "scales", torch.int16, rows * (cols // 64)),
                                   _dev(biases, "biases", torch.int16, rows * (cols // 64)), _stream())
    _status(rc, "tq_quantize_affine4")


def tq_repack_affine4(words: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, rows: int, cols: int,
                      qs: torch.Tensor, d: torch.Tensor) -> None:
    """MLX-layout affine 4-bit groups -> tiled layout (TQ_AFFINE4)."""
    _int("rows", rows, 0, I64[1])
    _int("cols", cols, 0, I64[1])
    qb, db = tq_qmat_bytes(TQ_AFFINE4, rows, cols)
    rc = lib().tq_repack_affine4(_dev(words, "words", torch.int32, rows * (cols // 8)),
                                 _dev(scales, "scales", torch.int16, rows * (cols // 64)),
                                 _dev(biases, "biases", torch.int16, rows * (cols // 64)), rows, cols,
                                 _dev(qs, "qs", torch.uint8, qb), _dev(d, "d", torch.int16, db // 2), _stream())
    _status(rc, "tq_repack_affine4")


def quantize_affine4(w: torch.Tensor):
    """f32 [rows][cols] (device) -> (words, scales, biases) in MLX's layout."""
    rows, cols = w.shape
    words = torch.empty(rows, cols // 8, dtype=torch.int32, device=w.device)
    scales = torch.empty(rows, cols // 64, dtype=torch.int16, device=w.device)
    biases = torch.empty(rows, cols // 64, dtype=torch.int16, device=w.device)
    tq_quantize_affine4(w.contiguous(), rows, cols, words, scales, biases)
    return words, scales, biases


# ----------------------------------------------------------------------------- matrices

class QMat:
    """One quantized matrix [rows][cols] in the tiled layout, in device memory (torch-owned)."""

    def __init__(self, wtype: int, rows: int, cols: int, qs: torch.Tensor, d: torch.Tensor):
        self.wtype, self.rows, self.cols, self.qs, self.d = wtype, rows, cols, qs, d

    @property
    def abi(self) -> TqQmat:
        return TqQmat(self.qs.data_ptr(), self.d.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.qs.numel() + 2 * self.d.numel()

    @classmethod
    def empty(cls, wtype: int, rows: int, cols: int, device) -> "QMat":
        qb, db = tq_qmat_bytes(wtype, rows, cols)
        qs = torch.empty(qb, dtype=torch.uint8, device=device)
        d = torch.empty(db // 2, dtype=torch.int16, device=device)
        return cls(wtype, rows, cols, qs, d)

    @classmethod
    def from_blocks(cls, wtype: int, blocks: torch.Tensor, rows: int, cols: int) -> "QMat":
        """GGUF-order block bytes (device uint8, [rows][cols/32][34|18]) -> tiled layout."""
        m = cls.empty(wtype, rows, cols, blocks.device)
        tq_repack(wtype, blocks, rows, cols, m.qs, m.d)
        return m


def quantize(w: torch.Tensor, wtype: int) -> torch.Tensor:
    """f32 [rows][cols] (device) -> GGUF-order blocks uint8 [rows][cols/32][34|18]."""
    rows, cols = w.shape
    out = torch.empty(rows, cols // 32, BLOCK_BYTES[wtype], dtype=torch.uint8, device=w.device)
    tq_quantize(wtype, w.contiguous(), rows, cols, out)
    return out


def tq_dequantize(m: QMat, row0: int = 0, n_rows: Optional[int] = None,
                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    n_rows = m.rows - row0 if n_rows is None else n_rows
    _int("row0", row0, 0, m.rows)
    _int("n_rows", n_rows, 0, m.rows - row0)
    if out is None:
        out = torch.empty(n_rows, m.cols, dtype=torch.float32, device=m.qs.device)
    rc = lib().tq_dequantize(m.wtype, m.abi, m.cols, row0, n_rows,
                             _dev(out, "out", torch.float32, n_rows * m.cols), _stream())
    _status(rc, "tq_dequantize")
    return out


def tq_gemv(m: QMat, x: torch.Tensor, residual: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y[b] = residual[b] + W x[b] for x [batch][cols] f32."""
    x2 = x.reshape(-1, m.cols)
    B = _int("batch", x2.shape[0], 1, I32[1])
    if out is None:
        out = torch.empty(B, m.rows, dtype=torch.float32, device=x.device)
    rc = lib().tq_gemv(m.wtype, m.abi, m.rows, m.cols, _dev(x2, "x", torch.float32, B * m.cols), B,
                       _dev(residual, "residual", torch.float32, B * m.rows),
                       _dev(out, "y", torch.float32, B * m.rows), _stream())
    _status(rc, "tq_gemv")
    return out


def tq_gemm(m: QMat, x: torch.Tensor, residual: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None, scratch: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y[t] = residual[t] + W x[t] for x [n_rows][cols] f32: the GEMM of
    prefill and batched decode.  `scratch`: optional uint8 device buffer of at
    least tq_gemm_scratch_bytes(rows, n_rows, cols) + 256 bytes, reused across
    calls (calls on it must not overlap)."""
    x2 = x.reshape(-1, m.cols)
    T = _int("n_rows", x2.shape[0], 1, I32[1])
    nb = int(lib().tq_gemm_scratch_bytes(m.rows, T, m.cols))
    if nb == 0:
        raise TqError(f"tq_gemm: unsupported shape ({T}, {m.cols})")
    if scratch is None:
        scratch = torch.empty(nb + 256, dtype=torch.uint8, device=x.device)
    elif scratch.numel() < nb + 256:
        raise TqError(f"scratch holds {scratch.numel()} bytes, needs {nb + 256}")
    off = (-scratch.data_ptr()) % 256
    if out is None:
        out = torch.empty(T, m.rows, dtype=torch.float32, device=x.device)
    rc = lib().tq_gemm(m.wtype, m.abi, m.rows, m.cols, _dev(x2, "x", torch.float32, T * m.cols), T,
                       _dev(residual, "residual", torch.float32, T * m.rows),
                       _dev(out, "y", torch.float32, T * m.rows),
                       ctypes.c_void_p(scratch.data_ptr() + off), _stream())
    _status(rc, "tq_gemm")
    return out


def tq_swiglu_gemv(gate: QMat, up: QMat, x: torch.Tensor, gain: Optional[torch.Tensor] = None,
                   eps: float = 1e-6, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """silu(Wg h) * (Wu h) with h = rms_norm(x, gain) (or x when gain is None)."""
    x2 = x.reshape(-1, gate.cols)
    B = _int("batch", x2.shape[0], 1, I32[1])
    if out is None:
        out = torch.empty(B, gate.rows, dtype=torch.float32, device=x.device)
    rc = lib().tq_swiglu_gemv(gate.wtype, gate.abi, up.abi, gate.rows, gate.cols,
                              _dev(x2, "x", torch.float32, B * gate.cols), B,
                              _dev(gain, "gain", torch.float32, gate.cols), float(eps),
                              _dev(out, "out", torch.float32, B * gate.rows), _stream())
    _status(rc, "tq_swiglu_gemv")
    return out


def tq_lm_head(m: QMat, x: torch.Tensor, gain: torch.Tensor, eps: float = 1e-6,
               want_logits: bool = True):
    """(logits [batch][vocab] or None, argmax [batch] int32) of rms_norm(x) through W."""
    x2 = x.reshape(-1, m.cols)
    B = _int("batch", x2.shape[0], 1, I32[1])
    logits = torch.empty(B, m.rows, dtype=torch.float32, device=x.device) if want_logits else None
    am = torch.empty(B, dtype=torch.int32, device=x.device)
    scratch = torch.empty(B, dtype=torch.int64, device=x.device)
    rc = lib().tq_lm_head(m.wtype, m.abi, m.rows, m.cols, _dev(x2, "x", torch.float32), B,
                          _dev(gain, "gain", torch.float32, m.cols), float(eps),
                          _dev(logits, "logits", torch.float32), _dev(am, "argmax", torch.int32),
                          _dev(scratch, "scratch", torch.int64), _stream())
    _status(rc, "tq_lm_head")
    return logits, am


def tq_sample(logits: torch.Tensor, temperature: torch.Tensor, top_p: torch.Tensor, u: torch.Tensor,
              out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Temperature / top-p sampling of logits [batch][vocab] on the device:
    per row a temperature (0: greedy), a top_p and a uniform number u in
    [0, 1) (f32 device tensors of [batch]); returns int32 token ids."""
    lg = logits.reshape(-1, logits.shape[-1])
    B = _int("batch", lg.shape[0], 1, I32[1])
    V = _int("vocab", lg.shape[1], 1, 1 << 24)
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=lg.device)
    rc = lib().tq_sample(_dev(lg, "logits", torch.float32, B * V), B, V,
                         _dev(temperature, "temperature", torch.float32, B), _dev(top_p, "top_p", torch.float32, B),
                         _dev(u, "u", torch.float32, B), _dev(out, "out", torch.int32, B), _stream())
    _status(rc, "tq_sample")
    return out


def tq_lm_head_static(m: QMat, x: torch.Tensor, gain: torch.Tensor, eps: float = 1e-6,
                      want_logits: bool = True, logits: Optional[torch.Tensor] = None,
                      argmax: Optional[torch.Tensor] = None):
    """tq_lm_head without caller scratch, for callers that cannot allocate
    device memory: the argmax keys live in a static device array inside the
    library (at most LM_HEAD_STATIC_MAX_BATCH rows).  Pass preallocated
    `logits` / `argmax` to keep the call itself free of allocations.  Calls
    that overlap on the GPU race on the shared array."""
    x2 = x.reshape(-1, m.cols)
    B = _int("batch", x2.shape[0], 1, LM_HEAD_STATIC_MAX_BATCH)
    if logits is None and want_logits:
        logits = torch.empty(B, m.rows, dtype=torch.float32, device=x.device)
    if argmax is None:
        argmax = torch.empty(B, dtype=torch.int32, device=x.device)
    rc = lib().tq_lm_head_static(m.wtype, m.abi, m.rows, m.cols, _dev(x2, "x", torch.float32), B,
                                 _dev(gain, "gain", torch.float32, m.cols), float(eps),
                                 _dev(logits, "logits", torch.float32, B * m.rows),
                                 _dev(argmax, "argmax", torch.int32, B), _stream())
    _status(rc, "tq_lm_head_static")
    return logits, argmax


# ----------------------------------------------------------------------------- model

LAYER_MATS = ("attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up", "ffn_down")
LAYER_GAINS = ("attn_norm", "ffn_norm", "attn_q_norm", "attn_k_norm")
LAYER_BIASES = ("attn_q_bias", "attn_k_bias", "attn_v_bias")
ARCHS = {"qwen3": 0, "llama": 1, "qwen2": 2, "gemma3": 3}


class Model:
    """A decoder over tiled quantized weights, a torch-allocated workspace and
    KV cache.  ``mats`` maps GGUF-style names (``token_embd``,
    ``blk.{i}.attn_q`` ...; optionally ``output``) to QMat; ``gains`` maps
    ``blk.{i}.attn_norm`` ... and ``output_norm`` (and for qwen2 the biases
    ``blk.{i}.attn_{q,k,v}_bias``) to f32 device tensors.  ``arch`` names the
    layer recipe: qwen3, llama, qwen2 or gemma3 (with ``sliding_window``,
    ``sliding_pattern`` and ``logit_softcap``)."""

    def __init__(self, *, vocab, hidden, n_layers, n_heads, n_kv_heads, head_dim, ffn,
                 wtype, kv, mats: dict, gains: dict, max_batch=1, max_ctx=4096,
                 max_prefill=512, page_size=0, n_pages=0, rms_eps=1e-6, rope_theta=1e6,
                 device="cuda", arch="qwen3", sliding_window=0, sliding_pattern=0, logit_softcap=0.0):
        self._handle = None
        self._thread = threading.get_ident()
        wt = WTYPES[wtype] if isinstance(wtype, str) else wtype
        kvt = {"f32": TQ_KV_F32, "f16": TQ_KV_F16}[kv] if isinstance(kv, str) else kv
        if arch not in ARCHS:
            raise TqError(f"arch must be one of {sorted(ARCHS)} (got {arch!r})")
        self.arch = arch
        vals = dict(vocab=vocab, hidden=hidden, n_layers=n_layers, n_heads=n_heads,
                    n_kv_heads=n_kv_heads, head_dim=head_dim, ffn=ffn, max_batch=max_batch,
                    max_ctx=max_ctx, max_prefill=max_prefill, page_size=page_size,
                    n_pages=n_pages, sliding_window=sliding_window, sliding_pattern=sliding_pattern)
        for k, v in vals.items():
            _int(k, v, 0, I32[1])
        self.cfg = TqConfig(rms_eps=float(rms_eps), rope_theta=float(rope_theta), wtype=wt,
                            kvtype=kvt, arch=ARCHS[arch], logit_softcap=float(logit_softcap), **vals)
        self.device = torch.device(device)
        if self.device.type != "cuda" or (self.device.index is not None and
                                          self.device.index != torch.cuda.current_device()):
            raise TqError(f"the model's device {self.device} must be the current CUDA device "
                          f"(cuda:{torch.cuda.current_device()})")
        self.device = torch.device("cuda", torch.cuda.current_device())
        ws = tq_workspace_bytes(self.cfg)
        if ws == 0:
            raise TqError(f"invalid configuration: {tq_last_error()}")
        kvb = tq_kv_cache_bytes(self.cfg)
        self.workspace = torch.empty(ws + 256, dtype=torch.uint8, device=self.device)
        self._ws_off = (-self.workspace.data_ptr()) % 256
        elt = torch.float16 if kvt == TQ_KV_F16 else torch.float32
        esz = 2 if kvt == TQ_KV_F16 else 4
        self.k_cache = torch.zeros(kvb // esz, dtype=elt, device=self.device)
        self.v_cache = torch.zeros(kvb // esz, dtype=elt, device=self.device)
        self.mats, self.gains = mats, gains
        layers = (TqLayer * n_layers)()
        for i in range(n_layers):
            L = layers[i]
            for n in LAYER_MATS:
                setattr(L, n, mats[f"blk.{i}.{n}"].abi)
            for n in LAYER_GAINS + LAYER_BIASES:
                g = gains.get(f"blk.{i}.{n}")
                if g is not None:
                    setattr(L, n + "_dev", g.data_ptr())
        self._layers = layers
        out = mats.get("output")
        self._weights = TqWeights(mats["token_embd"].abi, out.abi if out is not None else TqQmat(0, 0),
                                  gains["output_norm"].data_ptr(),
                                  ctypes.cast(layers, ctypes.POINTER(TqLayer)))
        h = ctypes.c_void_p()
        rc = lib().tq_model_create(ctypes.byref(self.cfg), ctypes.byref(self._weights),
                                   ctypes.c_void_p(self.workspace.data_ptr() + self._ws_off),
                                   ctypes.c_void_p(self.k_cache.data_ptr()),
                                   ctypes.c_void_p(self.v_cache.data_ptr()), ctypes.byref(h))
        _status(rc, "tq_model_create")
        self._handle = h

    # -- handle discipline
    def __copy__(self):
        raise TypeError("Model owns a C handle and cannot be copied")

    __deepcopy__ = lambda self, memo: self.__copy__()  # noqa: E731

    def __reduce__(self):
        raise TypeError("Model owns a C handle and cannot be pickled")

    def _h(self) -> ctypes.c_void_p:
        if self._handle is None:
            raise TqError("model is closed")
        if threading.get_ident() != self._thread:
            raise TqError("model used from a thread other than the one that created it")
        return self._handle

    def _after(self, rc: int, what: str):
        if rc != TQ_OK and self._handle is not None and lib().tq_model_poisoned(self._handle):
            msg = tq_last_error()
            self.close()
            raise TqPoisoned(f"{what}: {msg}")
        _status(rc, what)

    def close(self):
        if self._handle is not None:
            if threading.get_ident() != self._thread:
                self._handle = None        # leak rather than free on a foreign thread
                raise TqError("close() from another thread: handle leaked")
            lib().tq_model_free(self._handle)
            self._handle = None

    def __del__(self):
        try:
            if self._handle is not None and threading.get_ident() == self._thread:
                lib().tq_model_free(self._handle)
                self._handle = None
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- work
    @property
    def launches_per_step(self) -> int:
        return int(lib().tq_decode_launches(self._h(), 1))

    def decode_launches(self, batch: int) -> int:
        """Kernel launches of one decode step of `batch` sequences."""
        return int(lib().tq_decode_launches(self._h(), batch))

    def prefill(self, tokens: torch.Tensor, start_pos: int = 0, seq: int = 0,
                block_table: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                argmax: Optional[torch.Tensor] = None) -> torch.Tensor:
        n = _int("n_tokens", tokens.numel(), 1, I32[1])
        _int("start_pos", start_pos, 0, I32[1])
        _int("seq", seq, 0, I32[1])
        if argmax is None:
            argmax = torch.empty(1, dtype=torch.int32, device=self.device)
        rc = lib().tq_prefill(self._h(), seq, _dev(tokens, "tokens", torch.int32), n, start_pos,
                              _dev(block_table, "block_table", torch.int32),
                              _dev(logits, "logits", torch.float32, self.cfg.vocab),
                              _dev(argmax, "argmax", torch.int32, 1), _stream(self.device))
        self._after(rc, "tq_prefill")
        return argmax

    def decode_step(self, tokens: torch.Tensor, positions: torch.Tensor, kv_lens: torch.Tensor,
                    block_table: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                    argmax: Optional[torch.Tensor] = None, graph: bool = False) -> torch.Tensor:
        B = _int("batch", tokens.numel(), 1, I32[1])
        if argmax is None:
            argmax = torch.empty(B, dtype=torch.int32, device=self.device)
        fn = lib().tq_decode_step_graph if graph else lib().tq_decode_step
        rc = fn(self._h(), B, _dev(tokens, "tokens", torch.int32, B),
                _dev(positions, "positions", torch.int32, B), _dev(kv_lens, "kv_lens", torch.int32, B),
                _dev(block_table, "block_table", torch.int32),
                _dev(logits, "logits", torch.float32, B * self.cfg.vocab),
                _dev(argmax, "argmax", torch.int32, B), _stream(self.device))
        self._after(rc, "tq_decode_step_graph" if graph else "tq_decode_step")
        return argmax

    def decode_chain(self, layer: int) -> None:
        """Enqueue the batch-1 decode step's GEMV chain after `layer`'s attention
        on its own (tq_decode_chain), over the workspace's current activations."""
        _int("layer", layer, 0, self.cfg.n_layers - 1)
        self._after(lib().tq_decode_chain(self._h(), layer, _stream(self.device)), "tq_decode_chain")

    def set_wait_limit(self, polls: int) -> None:
        """Polls after which a GEMV chain's grid-wide waits give up (0: the
        default); a tiny limit exercises the timeout path (tq_model_set_wait_limit)."""
        _int("polls", polls, 0, 2**32 - 1)
        self._after(lib().tq_model_set_wait_limit(self._h(), polls), "tq_model_set_wait_limit")

    def step(self, tokens: torch.Tensor, row_seq: torch.Tensor, row_pos: torch.Tensor, last_row: torch.Tensor,
             block_table: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
             argmax: Optional[torch.Tensor] = None) -> torch.Tensor:
        """One continuous-batching step (tq_step): token rows of several
        sequences (prompt chunks and decode tokens mixed); returns the greedy
        token of each sequence's `last_row`."""
        n = _int("n_rows", tokens.numel(), 1, I32[1])
        S = _int("n_seq", last_row.numel(), 1, I32[1])
        if argmax is None:
            argmax = torch.empty(S, dtype=torch.int32, device=self.device)
        rc = lib().tq_step(self._h(), n, _dev(tokens, "tokens", torch.int32, n),
                           _dev(row_seq, "row_seq", torch.int32, n), _dev(row_pos, "row_pos", torch.int32, n), S,
                           _dev(last_row, "last_row", torch.int32, S), _dev(block_table, "block_table", torch.int32),
                           _dev(logits, "logits", torch.float32, S * self.cfg.vocab),
                           _dev(argmax, "argmax", torch.int32, S), _stream(self.device))
        self._after(rc, "tq_step")
        return argmax

    def status(self) -> int:
        bits = ctypes.c_uint32(0)
        rc = lib().tq_model_status(self._h(), _stream(self.device), ctypes.byref(bits))
        if rc != TQ_OK:
            msg = tq_last_error()
            self.close()
            raise TqPoisoned(f"tq_model_status: {msg}")
        return int(bits.value)

    def weight_bytes(self) -> int:
        return sum(m.nbytes for m in self.mats.values())


def tq_model_create(*args, **kw) -> Model:
    return Model(*args, **kw)
