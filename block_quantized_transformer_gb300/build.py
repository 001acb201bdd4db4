"""Build libtq.so (the CUDA kernels and the C ABI of include/tq.h) in-tree.

Every translation unit is compiled by nvcc for sm_103a in parallel, then
linked into block_quantized_transformer_gb300/_build/libtq.so against the
shared CUDA runtime.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libtq.so")
SOURCES = ["api.cu", "quant.cu", "gemv.cu", "gemv_q4.cu", "gemv_q8.cu", "gemv_a4.cu", "tcgemm.cu", "attn.cu", "attn_prefill.cu", "sample.cu", "lm_head_static.cu"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def flags(arch: str) -> list:
    return ["-O3", "-std=c++17", f"-gencode=arch=compute_{arch},code=sm_{arch}", "-lineinfo",
            "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-I",
            os.path.join(ROOT, "include")]


def build(arch: str = "103a", verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc(), *flags(arch), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"--- {src}\n{out.decode(errors='replace')}")
    if errors:
        raise RuntimeError("libtq build failed:\n" + "\n".join(errors))
    tmp = LIB + ".tmp"
    cmd = [nvcc(), f"-gencode=arch=compute_{arch},code=sm_{arch}", "-shared", "-cudart", "shared",
           "-o", tmp, *objs, "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("libtq link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
