"""Compile the CUDA library libdit_attn.so in place (sm_103a only).

    python -m diffusion_transformer_joint_causal_b300.build [--force]
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "dit_attn.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "fmha_pair.cuh"),
                  os.path.join(CSRC, "rmsnorm.cuh"), os.path.join(CSRC, "combine.cuh"),
                  os.path.join(CSRC, "quantize.cuh"),
                  os.path.join(os.path.dirname(PKG), "include", "dit_attn.h")]
LIB = os.path.join(PKG, "libdit_attn.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-warn-spills"]


def build(force: bool = False, verbose: bool = False) -> str:
    stale = force or not os.path.exists(LIB) or any(
        os.path.getmtime(p) > os.path.getmtime(LIB) for p in DEPS)
    if stale:
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [NVCC, *FLAGS, *(["-Xptxas", "-v"] if verbose else []), *SOURCES, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
