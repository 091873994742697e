"""Compile the CPU oracle (test infrastructure) into oracle/_build/liboracle.so.

Flags keep the arithmetic exactly as written: no contraction of a*b+c into an
fma (GCC contracts by default on aarch64), no fast-math reassociation.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.cpp")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CXXFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17", "-fPIC", "-shared"]


def build(src: str = SRC, out: str = LIB, force: bool = False) -> str:
    """Compile ``src`` into the shared library ``out``; returns ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", *CXXFLAGS, src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
