"""Compile the C oracle into oracle/libdsa_oracle.so (gcc, OpenMP when available).

The oracle is test infrastructure; building it is part of the package build so
that the tests and the benchmark's CPU baseline find it on any machine.
``-ffp-contract=off`` keeps every fp64 multiply and add separately rounded, so
x86 and Arm hosts produce the same bits.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dsa_oracle.c")
LIB = os.path.join(HERE, "libdsa_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
            SRC, "-o", LIB + ".tmp", "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            if verbose:
                print(" ".join(cmd))
            return LIB
        if verbose:
            print(r.stderr, file=sys.stderr)
    raise RuntimeError("could not compile the oracle: " + r.stderr)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
