"""Build the CPU oracle shared library (test infrastructure only).

The oracle is plain C compiled with gcc; FP contraction is switched off so
that x86-64 and aarch64 hosts round every FP64 operation identically.
"""
from __future__ import annotations

import hashlib
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "libmoe_oracle.so")
STAMP = LIB + ".src-sha"


def _digest() -> str:
    with open(SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def build(force: bool = False) -> str:
    """Compile oracle/moe_oracle.c into oracle/libmoe_oracle.so (if stale)."""
    want = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == want:
                return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(want + "\n")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
