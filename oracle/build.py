"""Compile the C oracle (test infrastructure) into oracle/_lib/libhc_oracle.so.

Plain gcc, no architecture flags and no floating-point contraction, so x86 and
Arm hosts evaluate the same float64 expressions in the same order.
"""

from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hc_oracle.c")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libhc_oracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = LIB + ".tmp"
    try:
        subprocess.run(base + ["-fopenmp", SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime on this host: the oracle still builds, single-threaded.
        subprocess.run(base + [SRC, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
