"""Compile the C oracle into ``oracle/_build/libdg_oracle.so`` with gcc.

Test infrastructure only.  Plain C11, no fast-math and no FMA contraction,
so that the same source gives the same bits on x86-64 and AArch64.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dg_oracle.c")
HDR = os.path.join(HERE, "dg_oracle.h")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libdg_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off",
          "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False) -> str:
    """Build the oracle library if missing or out of date; return its path."""
    if force or _stale():
        os.makedirs(OUT_DIR, exist_ok=True)
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
