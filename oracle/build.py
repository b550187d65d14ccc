"""Build the oracle's shared library (test infrastructure only).

Compiles ``iha_oracle.c`` with the host C compiler and OpenMP into
``liboracle.so`` beside it.  Plain C, no architecture-specific flags, so it
builds the same on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "iha_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
