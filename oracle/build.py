"""Compile the CPU oracle (mp_oracle.c) into oracle/_mp_oracle.so with gcc.

Test infrastructure: the oracle is built next to its source so that the
tests, the smoke check and the benchmark's CPU baseline can load it. The
flags keep the arithmetic exactly as written: no FMA contraction (the only
fused operations are the explicit fmaf calls), no fast-math, strict C11.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mp_oracle.c")
HDR = os.path.join(HERE, "mp_oracle.h")
LIB = os.path.join(HERE, "_mp_oracle.so")

CFLAGS = [
    "-O2", "-std=c11", "-fPIC", "-shared",
    "-ffp-contract=off", "-fno-fast-math", "-fno-finite-math-only",
    "-Wall", "-Wextra", "-Werror",
]


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    lib_t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > lib_t for p in (SRC, HDR))


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its sources."""
    if force or is_stale():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
