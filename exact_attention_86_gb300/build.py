"""Builds the C-ABI library ``libattn.so`` in-tree with nvcc for sm_103a.

``python -m exact_attention_86_gb300.build`` (or ``build()``) compiles
``csrc/attn_fwd.cu`` (which includes the backward kernels of
``csrc/attn_bwd.cuh`` and the PTX wrappers of ``csrc/sm103_ptx.cuh``) into
``exact_attention_86_gb300/libattn.so``.  The library
links only the CUDA runtime (statically); the driver's tensor-map encoder is
looked up at run time, so the library also loads on a machine without a GPU.
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "attn_fwd.cu")]
DEPS = SOURCES + [os.path.join(PKG, "csrc", "sm103_ptx.cuh"), os.path.join(PKG, "csrc", "attn_bwd.cuh"),
                  os.path.join(ROOT, "include", "attn.h")]
LIB = os.path.join(PKG, "libattn.so")
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources; return its path."""
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= t for d in DEPS):
            return LIB
    cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", LIB + ".tmp", *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
