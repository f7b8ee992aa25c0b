"""Builds the C oracle (``pkv_oracle.c``) into ``oracle/_build/libpkv_oracle.so``.

Test infrastructure only: the oracle is the plain fp64 CPU definition the CUDA
library is checked against.  Plain gcc, OpenMP over (sequence, query head),
no architecture-specific flags, floating-point contraction off so x86 and Arm
hosts evaluate the same expressions.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpkv_oracle.so")


def build(force: bool = False) -> str:
    """Compiles the oracle if the shared object is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
