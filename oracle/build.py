"""Compile the C oracle into ``oracle/_build/libpa_oracle.so`` with gcc.

Test infrastructure only (see ``oracle/__init__.py``).  Plain C, OpenMP over
the outer (sequence, query head) loop when the compiler supports it, no
floating-point contraction so x86 and Arm hosts give the same bits.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa_oracle.so")


def build(force: bool = False, out: str | None = None, src: str | None = None) -> str:
    """Build the oracle library; return its path.  ``src``/``out`` let the
    tests compile deliberately broken copies of the oracle elsewhere."""
    src = src or SRC
    out = out or LIB
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wno-unknown-pragmas"]
    tmp = out + f".tmp{os.getpid()}"
    cmd = base + ["-fopenmp", "-o", tmp, src, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP runtime: build single-threaded
        cmd = base + ["-o", tmp, src, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{' '.join(cmd)}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
