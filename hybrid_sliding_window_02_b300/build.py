"""Build libswasink.so in-tree with nvcc for sm_103a (B300).

``python -m hybrid_sliding_window_02_b300.build`` (or ``build()``) compiles
``csrc/swasink.cu`` into ``libswasink.so`` next to this file.  Extra flags can be
passed through the environment variable ``SWASINK_NVCC_FLAGS``.
"""
from __future__ import annotations

import os
import shlex
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "swasink.cu")
LIB = os.path.join(HERE, "libswasink.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")


def _sources():
    csrc = os.path.join(HERE, "csrc")
    files = [os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".cuh"))]
    return files + [os.path.join(INCLUDE, "swasink.h")]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
           "-I", INCLUDE, SRC, "-o", tmp]
    cmd += shlex.split(os.environ.get("SWASINK_NVCC_FLAGS", ""))
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
