"""Build the CPU oracle (plain C) into oracle/_build/liboracle.so.

Test infrastructure: compiled by ``__graft_entry__.build()`` beside the CUDA
library so the tests and the benchmark's CPU-baseline leg can load it.  The
flags keep fp32 arithmetic exactly as written: no fast-math, no FMA
contraction (GCC contracts by default on aarch64).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-Wall", "-Wextra", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
