"""Builds libfp4idx.so (the CUDA kernels + C ABI) in-tree with nvcc for
sm_103a.  The library links the CUDA runtime statically, so it needs only the
NVIDIA driver at run time.

    python -m fp4_sparse_attention_fp4idx_gb300.build [--force] [-v]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRCS = [os.path.join(PKG, "csrc", name)
        for name in ("fp4idx.cu", "fp4idx_stream.cu", "fp4idx_scorer.cu", "fp4idx_host.cu")]
HDRS = [os.path.join(ROOT, "include", "fp4idx.h"), os.path.join(PKG, "csrc", "fp4idx_common.cuh")]
LIB = os.path.join(PKG, "libfp4idx.so")

# Bit-exact fp32: no FMA contraction, IEEE division/sqrt, subnormals kept.
NVCC_FLAGS = [
    "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfp4idx.so")


def build(force: bool = False, verbose: bool = False) -> str:
    newest = max(os.path.getmtime(f) for f in (*SRCS, *HDRS))
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    tag = f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in SRCS:  # one translation unit per process, compiled in parallel
        obj = os.path.join(PKG, os.path.basename(src) + tag + ".o")
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append((cmd, subprocess.Popen(cmd)))
    try:
        for cmd, proc in procs:
            if proc.wait() != 0:
                raise subprocess.CalledProcessError(proc.returncode, cmd)
        tmp = LIB + tag
        subprocess.run([nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs,
                        "-o", tmp], check=True)
        os.replace(tmp, LIB)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
