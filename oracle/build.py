"""Compile the CPU oracle (mp_oracle.c) into oracle/_mp_oracle.so with gcc,
and its command-line front end (mp_oracle_cli.c) into oracle/_mp_oracle_cli.

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
CLI_SRC = os.path.join(HERE, "mp_oracle_cli.c")
CLI = os.path.join(HERE, "_mp_oracle_cli")

CFLAGS = [
    "-O2", "-std=c11", "-fPIC", "-shared",
    "-ffp-contract=off", "-fno-fast-math", "-fno-finite-math-only",
    "-Wall", "-Wextra", "-Werror",
]


def _stale(out, sources) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in sources)


def is_stale() -> bool:
    return _stale(LIB, (SRC, HDR)) or _stale(CLI, (SRC, HDR, CLI_SRC))


def build(force: bool = False) -> str:
    """Build the oracle library (and its command-line front end) if missing
    or older than their sources."""
    if force or _stale(LIB, (SRC, HDR)):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, LIB)
    if force or _stale(CLI, (SRC, HDR, CLI_SRC)):
        tmp = CLI + f".tmp{os.getpid()}"
        flags = [f for f in CFLAGS if f not in ("-shared", "-fPIC")]
        subprocess.run(["gcc", *flags, SRC, CLI_SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, CLI)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
