"""Compile the CPU oracle (test infrastructure) into ``oracle/liboracle.so``.

Plain gcc, no fast-math, no contraction into fused multiply-add (GCC contracts by
default on aarch64), no auto-vectorisation, so that every fp32 operation in
``lema_oracle.c`` is one IEEE operation rounded to nearest even.  OpenMP is used
when the compiler has it; it only splits the loops over independent elements (or
8-bit blocks) across threads.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lema_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
              "-fno-tree-vectorize", "-fPIC", "-shared", "-Wall"]


def compile_oracle(src: str = SRC, out: str = LIB, extra: list[str] | None = None) -> str:
    """Compile ``src`` into the shared library ``out``; returns ``out``."""
    extra = list(extra or [])
    cmd = ["gcc", *BASE_FLAGS, "-fopenmp", *extra, src, "-o", out, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        # A toolchain without OpenMP still builds the single-threaded oracle.
        cmd = ["gcc", *BASE_FLAGS, *extra, src, "-o", out, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    return out


def ensure_built() -> str:
    """Build the oracle if the library is missing or older than its source."""
    if (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        compile_oracle()
    return LIB


if __name__ == "__main__":
    print(compile_oracle())
    sys.exit(0)
