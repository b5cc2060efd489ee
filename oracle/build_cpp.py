"""Compile the C++ oracle (lidx_oracle.cpp) into liblidx_oracle.so next to it.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain g++ with OpenMP;
no CUDA header, no source shared with the GPU library.  IEEE arithmetic is
kept as written: no -ffast-math, and -ffp-contract=off so that no multiply and
add are fused into one rounding.  Rebuilds only when the source is newer.
"""

from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lidx_oracle.cpp")
LIB = os.path.join(HERE, "liblidx_oracle.so")
FLAGS = ["-O3", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = os.environ.get("CXX") or shutil.which("g++") or "g++"
    tmp = LIB + f".{os.getpid()}.tmp"
    r = subprocess.run([cxx, *FLAGS, "-fopenmp", SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the C++ oracle failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
