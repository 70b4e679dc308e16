"""Compile the C++ oracle (oracle/csrc/*.cpp) into oracle/liboracle.so (g++, C++17, OpenMP).

Plain host code: no architecture flags, and no fused multiply-adds formed by the compiler
(-ffp-contract=off), so the oracle rounds the same way on every machine it is built on.
"""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "liboracle.so")
FLAGS = ["-O3", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    sources = sorted(glob.glob(os.path.join(SRC, "*.cpp")))
    deps = sources + sorted(glob.glob(os.path.join(SRC, "*.h")))
    newest = max(os.path.getmtime(p) for p in deps)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [os.environ.get("CXX", "g++"), *FLAGS, "-o", tmp, *sources]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
