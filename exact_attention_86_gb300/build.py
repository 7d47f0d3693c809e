"""Builds the C-ABI library ``libattn.so`` in-tree with nvcc for sm_103a.

``python -m exact_attention_86_gb300.build`` (or ``build()``) compiles
``csrc/attn_fwd.cu`` (the one-tile forward kernels, the backward kernels of
``csrc/attn_bwd.cuh`` and the C ABI) and ``csrc/attn_fwd_pair.cu`` (the
two-tile forward kernel) in parallel, then links them into
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
SOURCES = [os.path.join(PKG, "csrc", "attn_fwd.cu"), os.path.join(PKG, "csrc", "attn_fwd_pair.cu")]
DEPS = SOURCES + [os.path.join(PKG, "csrc", n) for n in ("sm103_ptx.cuh", "attn_bwd.cuh", "attn_common.cuh",
                                                         "attn_pair_host.h")] + [os.path.join(ROOT, "include", "attn.h")]
LIB = os.path.join(PKG, "libattn.so")
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC"]


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
    objs = [LIB + "." + os.path.splitext(os.path.basename(src))[0] + ".o" for src in SOURCES]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, proc in procs if proc.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    subprocess.run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", LIB + ".tmp", *objs],
                   check=True)
    for obj in objs:
        os.remove(obj)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
