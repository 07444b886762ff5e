"""Compile the CPU oracle (test infrastructure) into oracle/liboracle.so with gcc.

The oracle is plain C11 with no CUDA header; it builds the same way on x86-64 and
aarch64.  Contraction of a*b+c into fused multiply-adds is switched off so that the
only fused multiply-adds are the explicit fmaf() calls of the EMA update.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spin_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    deps = [SRC, os.path.join(HERE, "spin_oracle.h")]
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(p) for p in deps):
            return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
