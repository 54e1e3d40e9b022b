"""Compile the CPU oracle (plain C, OpenMP) into oracle/_build/liboracle.so.

Test infrastructure: the library it builds is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

# IEEE single precision, one rounding per operation: no contraction of a*b+c
# into an FMA and no fast-math, so the fp32 decision steps are reproducible.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-fPIC", "-shared", "-Wall", "-Wno-unknown-pragmas"]


# "compiled" or "reused": what the last build() call did
last_action = None


def build(force: bool = False) -> str:
    global last_action
    src = os.path.join(HERE, "oracle.c")
    hdr = os.path.join(HERE, "oracle.h")
    os.makedirs(OUT_DIR, exist_ok=True)
    inputs = (src, hdr, os.path.abspath(__file__))  # the flags live in this file
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(f) for f in inputs)):
        last_action = "reused"
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    last_action = "compiled"
    return LIB


if __name__ == "__main__":
    print(build(force=True))
