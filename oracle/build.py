"""Build the CPU oracle (test infrastructure) into oracle/liboracle.so with gcc.

Only the tests, the smoke check and the benchmark's CPU-baseline leg load the
result.  Plain C99, -O2, no fast-math (IEEE single-precision division and
subtraction are part of the quantiser's definition), OpenMP for row-parallel
loops.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "w4a16_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["gcc", "-O2", "-std=c99", "-Wall", "-Wextra", "-fno-fast-math", "-ffp-contract=off",
           "-fopenmp", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp", "-lm"]
    subprocess.check_call(cmd)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
