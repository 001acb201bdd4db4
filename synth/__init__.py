"""Seeded synthetic inputs shared by the oracle and the GPU path.

This module holds no arithmetic of the decode method.  It describes the
workloads (sizes, seeds, formats) and turns (seed, stream, element index) into
numbers with one counter-based generator, Philox4x32-10 (Salmon et al., SC'11),
so that every element of every synthetic tensor can be produced on its own:

* ``philox4x32_10`` / ``normal`` / ``uniform_below`` -- plain NumPy versions
  (the readable definition, used on small cases and to pin the others);
* ``host_normal`` / ``host_uniform_below`` -- the same generator in C
  (``philox_ih.h`` + ``host.c``), multi-threaded, for large host tensors;
* ``dev_normal`` / ``dev_uniform_below`` -- the same generator as CUDA
  kernels (``device.cu``) writing into device memory.

"N(0, sigma)" is realised as an Irwin-Hall sum of eight 16-bit uniforms,
centred and scaled to standard deviation sigma: mean 0, the stated variance,
kurtosis -0.15, support +-4.9 sigma.  The sum is an exact integer and the
scaling one f32 multiply, so all three versions agree bit for bit.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")

MASK32 = np.uint64(0xFFFFFFFF)
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)
IH8_MEAN = 262140
IH8_SD = math.sqrt(8.0 * (65536.0 * 65536.0 - 1.0) / 12.0)

# Fixed stream ids: tensors of a model are numbered in this order, the
# prompt of sequence b uses PROMPT_STREAM + b, ragged lengths LENGTH_STREAM.
LAYER_TENSORS = ("attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up",
                 "ffn_down", "attn_norm", "ffn_norm", "attn_q_norm", "attn_k_norm")
BIAS_TENSORS = ("attn_q_bias", "attn_k_bias", "attn_v_bias")  # qwen2 only
PROMPT_STREAM = 1_000_000
LENGTH_STREAM = 2_000_000
KV_STREAM = 3_000_000
BIAS_STREAM = 4_000_000   # + 3 * layer + index in BIAS_TENSORS
WEIGHT_SIGMA = 0.02
BIAS_SIGMA = 0.1
ARCHS = ("qwen3", "llama", "qwen2", "gemma3")


def normal_scale(sigma: float) -> np.float32:
    """f32 factor turning a centred Irwin-Hall(8) integer into N(0, sigma)."""
    return np.float32(sigma / IH8_SD)


# ----------------------------------------------------------------------------
# NumPy definition of the generator
# ----------------------------------------------------------------------------

def philox4x32_10(ctr, key):
    """Philox4x32-10 on arrays: ctr = 4 arrays of uint32 values, key = (k0, k1)."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & MASK32 for c in ctr)
    k0 = np.asarray(key[0], dtype=np.uint64) & MASK32
    k1 = np.asarray(key[1], dtype=np.uint64) & MASK32
    for r in range(10):
        if r:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def words(seed: int, stream: int, idx) -> tuple:
    idx = np.asarray(idx, dtype=np.uint64)
    z = np.zeros_like(idx)
    return philox4x32_10((idx & MASK32, idx >> np.uint64(32), z, z), (seed, stream))


def ih8_centred(w) -> np.ndarray:
    s = np.zeros(np.shape(w[0]), dtype=np.int64)
    for wi in w:
        wi = wi.astype(np.int64)
        s += (wi & 0xFFFF) + (wi >> 16)
    return s - IH8_MEAN


def normal(seed: int, stream: int, n: int, first: int = 0, sigma: float = WEIGHT_SIGMA,
           mean: float = 0.0) -> np.ndarray:
    idx = np.arange(first, first + n, dtype=np.uint64)
    v = ih8_centred(words(seed, stream, idx)).astype(np.float32) * normal_scale(sigma)
    if mean != 0.0:
        v = np.float32(mean) + v
    return v.astype(np.float32)


def uniform_below(seed: int, stream: int, n: int, bound: int, first: int = 0) -> np.ndarray:
    idx = np.arange(first, first + n, dtype=np.uint64)
    w0 = words(seed, stream, idx)[0]
    return ((w0 * np.uint64(bound)) >> np.uint64(32)).astype(np.int32)


# ----------------------------------------------------------------------------
# Compiled versions (host C and CUDA)
# ----------------------------------------------------------------------------

HOST_LIB = os.path.join(_BUILD, "libtqs_host.so")
DEV_LIB = os.path.join(_BUILD, "libtqs_dev.so")


def build(device: bool = True, arch: str = "103a") -> None:
    """Compile the host generator (gcc) and, if asked, the device one (nvcc)."""
    os.makedirs(_BUILD, exist_ok=True)
    procs = [subprocess.Popen(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               os.path.join(_HERE, "host.c"), "-o", HOST_LIB])]
    if device:
        procs.append(subprocess.Popen(
            ["nvcc", "-O3", f"-gencode=arch=compute_{arch},code=sm_{arch}", "-shared",
             "-Xcompiler", "-fPIC", "-o", DEV_LIB, os.path.join(_HERE, "device.cu")]))
    for p in procs:
        if p.wait() != 0:
            raise RuntimeError("synth: build failed")


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            build(device=False)
        lib = ctypes.CDLL(HOST_LIB)
        lib.tqs_host_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                             ctypes.c_uint32, ctypes.c_uint32, ctypes.c_float,
                                             ctypes.c_float]
        lib.tqs_host_fill_uniform_below.argtypes = [ctypes.c_void_p, ctypes.c_uint64,
                                                    ctypes.c_uint64, ctypes.c_uint32,
                                                    ctypes.c_uint32, ctypes.c_uint32]
        lib.tqs_host_philox.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32,
                                        ctypes.c_void_p]
        _host = lib
    return _host


def host_philox(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _host_lib().tqs_host_philox(c.ctypes.data, key[0], key[1], out.ctypes.data)
    return out


def host_normal(seed: int, stream: int, n: int, first: int = 0, sigma: float = WEIGHT_SIGMA,
                mean: float = 0.0, out: Optional[np.ndarray] = None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _host_lib().tqs_host_fill_normal(out.ctypes.data, n, first, seed, stream,
                                     float(normal_scale(sigma)), float(mean))
    return out


def host_uniform_below(seed: int, stream: int, n: int, bound: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _host_lib().tqs_host_fill_uniform_below(out.ctypes.data, n, first, seed, stream, bound)
    return out


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError("synth: device generator not built (run synth.build())")
        lib = ctypes.CDLL(DEV_LIB)
        lib.tqs_dev_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_float,
                                            ctypes.c_float, ctypes.c_void_p]
        lib.tqs_dev_fill_uniform_below.argtypes = [ctypes.c_void_p, ctypes.c_uint64,
                                                   ctypes.c_uint64, ctypes.c_uint32,
                                                   ctypes.c_uint32, ctypes.c_uint32,
                                                   ctypes.c_void_p]
        _dev = lib
    return _dev


def dev_normal(out, seed: int, stream: int, first: int = 0, sigma: float = WEIGHT_SIGMA,
               mean: float = 0.0):
    """Fill the contiguous f32 CUDA tensor ``out`` on torch's current stream."""
    import torch
    assert out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
    st = torch.cuda.current_stream(out.device).cuda_stream
    rc = _dev_lib().tqs_dev_fill_normal(out.data_ptr(), out.numel(), first, seed, stream,
                                        float(normal_scale(sigma)), float(mean), st)
    if rc != 0:
        raise RuntimeError(f"synth: device fill failed ({rc})")
    return out


def dev_uniform_below(out, seed: int, stream: int, bound: int, first: int = 0):
    import torch
    assert out.is_cuda and out.dtype == torch.int32 and out.is_contiguous()
    st = torch.cuda.current_stream(out.device).cuda_stream
    rc = _dev_lib().tqs_dev_fill_uniform_below(out.data_ptr(), out.numel(), first, seed, stream,
                                               bound, st)
    if rc != 0:
        raise RuntimeError(f"synth: device fill failed ({rc})")
    return out


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """Sizes, formats and seeds of one synthetic decode workload."""
    name: str
    vocab: int
    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    wtype: str            # "q8_0" or "q4_0"
    kv: str               # "f32" or "f16"
    seed: int
    batch: int = 1
    prompt_len: int = 8
    decode_steps: int = 16
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    paged: bool = False
    page_size: int = 64
    ctx_lo: int = 0       # ragged batched mix: context lengths uniform in [ctx_lo, ctx_hi]
    ctx_hi: int = 0
    length_seed: int = 0
    # architecture of the decoder (which tensors exist; the oracle and the
    # library each read what it means): qwen3, llama (no per-head Q/K norm),
    # qwen2 (llama + Q/K/V biases), gemma3 (sliding window on a layer
    # pattern, tanh-approximated GELU in the gated FFN, final logit softcap)
    arch: str = "qwen3"
    sliding_window: int = 0
    sliding_pattern: int = 0
    logit_softcap: float = 0.0

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    def stream_of(self, name: str) -> int:
        """Generator stream of a tensor, by its GGUF-style name."""
        if name == "token_embd":
            return 0
        if name == "output_norm":
            return 1 + len(LAYER_TENSORS) * self.n_layers
        parts = name.split(".")
        assert parts[0] == "blk" and len(parts) == 3, name
        if parts[2] in BIAS_TENSORS:
            return BIAS_STREAM + 3 * int(parts[1]) + BIAS_TENSORS.index(parts[2])
        return 1 + len(LAYER_TENSORS) * int(parts[1]) + LAYER_TENSORS.index(parts[2])

    def matrix_shape(self, name: str) -> tuple:
        """[out, in] of a weight matrix (blocks run along `in`)."""
        H, hd = self.hidden, self.head_dim
        if name == "token_embd":
            return (self.vocab, H)
        kind = name.split(".")[-1]
        return {"attn_q": (self.n_heads * hd, H), "attn_k": (self.n_kv_heads * hd, H),
                "attn_v": (self.n_kv_heads * hd, H), "attn_output": (H, self.n_heads * hd),
                "ffn_gate": (self.ffn, H), "ffn_up": (self.ffn, H),
                "ffn_down": (H, self.ffn)}[kind]

    def gain_len(self, name: str) -> int:
        kind = name.split(".")[-1]
        return self.head_dim if kind in ("attn_q_norm", "attn_k_norm") else self.hidden

    def bias_len(self, name: str) -> int:
        kind = name.split(".")[-1]
        return (self.n_heads if kind == "attn_q_bias" else self.n_kv_heads) * self.head_dim

    def matrices(self) -> list:
        out = ["token_embd"]
        for i in range(self.n_layers):
            out += [f"blk.{i}.{t}" for t in LAYER_TENSORS[:7]]
        return out

    def gains(self) -> list:
        kinds = LAYER_TENSORS[7:] if self.arch in ("qwen3", "gemma3") else LAYER_TENSORS[7:9]
        out = []
        for i in range(self.n_layers):
            out += [f"blk.{i}.{t}" for t in kinds]
        return out + ["output_norm"]

    def biases(self) -> list:
        if self.arch != "qwen2":
            return []
        return [f"blk.{i}.{t}" for i in range(self.n_layers) for t in BIAS_TENSORS]

    def weight_count(self) -> int:
        return sum(int(np.prod(self.matrix_shape(m))) for m in self.matrices())

    def block_bytes(self) -> int:
        return 34 if self.wtype == "q8_0" else 18

    def prompt(self, b: int = 0, n: Optional[int] = None) -> np.ndarray:
        return uniform_below(self.seed, PROMPT_STREAM + b, n or self.prompt_len, self.vocab)

    def context_lengths(self) -> np.ndarray:
        span = self.ctx_hi - self.ctx_lo + 1
        return (self.ctx_lo + uniform_below(self.length_seed, LENGTH_STREAM, self.batch, span)
                ).astype(np.int32)


TINY = Workload("tiny_q8_0", vocab=4096, hidden=256, n_layers=2, n_heads=4, n_kv_heads=2,
                head_dim=64, ffn=768, wtype="q8_0", kv="f32", seed=0, prompt_len=8,
                decode_steps=16)
QWEN3_0P6B_Q8 = Workload("qwen3_0.6b_q8_0", vocab=151936, hidden=1024, n_layers=28, n_heads=16,
                         n_kv_heads=8, head_dim=128, ffn=3072, wtype="q8_0", kv="f32", seed=1,
                         prompt_len=128, decode_steps=128)
QWEN3_0P6B_Q4_LONG = Workload("qwen3_0.6b_q4_0_long", vocab=151936, hidden=1024, n_layers=28,
                              n_heads=16, n_kv_heads=8, head_dim=128, ffn=3072, wtype="q4_0",
                              kv="f16", seed=1, prompt_len=4096, decode_steps=256)
QWEN3_8B_Q4 = Workload("qwen3_8b_q4_0", vocab=151936, hidden=4096, n_layers=36, n_heads=32,
                       n_kv_heads=8, head_dim=128, ffn=12288, wtype="q4_0", kv="f16", seed=2,
                       prompt_len=2048, decode_steps=256)
QWEN3_8B_Q4_BATCHED = Workload("qwen3_8b_q4_0_batched32_paged", vocab=151936, hidden=4096,
                               n_layers=36, n_heads=32, n_kv_heads=8, head_dim=128, ffn=12288,
                               wtype="q4_0", kv="f16", seed=2, batch=32, prompt_len=2048,
                               decode_steps=128, paged=True, page_size=64, ctx_lo=512,
                               ctx_hi=8192, length_seed=3)
WORKLOADS = [TINY, QWEN3_0P6B_Q8, QWEN3_0P6B_Q4_LONG, QWEN3_8B_Q4, QWEN3_8B_Q4_BATCHED]

# Sibling architectures on the tiny shape (parity cases): the same sizes and
# seed as TINY, another layer recipe.
TINY_LLAMA = Workload("tiny_llama", vocab=4096, hidden=256, n_layers=2, n_heads=4, n_kv_heads=2,
                      head_dim=64, ffn=768, wtype="q8_0", kv="f32", seed=0, prompt_len=8,
                      decode_steps=16, arch="llama")
TINY_QWEN2 = Workload("tiny_qwen2", vocab=4096, hidden=256, n_layers=2, n_heads=4, n_kv_heads=2,
                      head_dim=64, ffn=768, wtype="q8_0", kv="f32", seed=0, prompt_len=8,
                      decode_steps=16, arch="qwen2")
TINY_GEMMA3 = Workload("tiny_gemma3", vocab=4096, hidden=256, n_layers=4, n_heads=4, n_kv_heads=2,
                       head_dim=64, ffn=768, wtype="q8_0", kv="f32", seed=0, prompt_len=8,
                       decode_steps=16, arch="gemma3", sliding_window=6, sliding_pattern=2,
                       logit_softcap=0.5)
ARCH_WORKLOADS = [TINY_LLAMA, TINY_QWEN2, TINY_GEMMA3]


def host_tensor(w: Workload, name: str, rows: Optional[slice] = None) -> np.ndarray:
    """A synthetic weight (f32, [out, in] row-major) or gain (f32), on the host.

    Matrices are N(0, 0.02); gains are 1 + N(0, 0.02); biases N(0, 0.1).
    ``rows`` selects a contiguous row range of a matrix without generating
    the rest.
    """
    stream = w.stream_of(name)
    if name.split(".")[-1] in BIAS_TENSORS:
        return host_normal(w.seed, stream, w.bias_len(name), sigma=BIAS_SIGMA)
    if name == "output_norm" or name.split(".")[-1] in LAYER_TENSORS[7:]:
        return host_normal(w.seed, stream, w.gain_len(name), mean=1.0)
    n_out, n_in = w.matrix_shape(name)
    r0, r1 = (0, n_out) if rows is None else (rows.start or 0, rows.stop or n_out)
    return host_normal(w.seed, stream, (r1 - r0) * n_in, first=r0 * n_in).reshape(r1 - r0, n_in)
