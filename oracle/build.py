"""Compile the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, no CUDA. -ffp-contract=off keeps every a*b+c as two roundings, which the
oracle's single-precision op order depends on (tests probe it).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "psadam_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    hdr = os.path.join(HERE, "psadam_oracle.h")
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(SRC), os.path.getmtime(hdr), os.path.getmtime(__file__))
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
