"""Builds the CPU oracle (``vs_oracle.c``) into ``oracle/_build/liboracle.so``.

Test infrastructure: only the test suite, the package smoke check and the
benchmark's CPU-baseline leg load the result.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vs_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= os.path.getmtime(SRC):
        return OUT
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = OUT + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, SRC, "-lm"]
    try:
        subprocess.check_call(base[:2] + ["-fopenmp"] + base[2:])
    except subprocess.CalledProcessError:
        subprocess.check_call(base)  # no OpenMP runtime: single-threaded oracle
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
