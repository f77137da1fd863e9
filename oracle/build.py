"""Compile the plain-C oracle into oracle/liboracle.so.

Test infrastructure only.  Flags: ISO C11, -O2, no contraction of a*b+c into a fused
multiply-add (aarch64 GCC fuses by default in GNU mode), no fast-math, so every fp32
operation rounds once and subnormals are kept.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = [
    "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fno-associative-math",
    "-fno-reciprocal-math", "-fPIC", "-shared", "-Wall", "-Wextra",
]


def build(force: bool = False) -> str:
    """Build liboracle.so if missing or older than oracle.c; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
