"""Compile the C oracle into ``oracle/_build/liboracle.so``.

Test infrastructure: the oracle is built so the tests, the smoke check and the
CPU-baseline leg of the benchmark can call it; nothing on the product path
links or loads it.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qmv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

# -ffp-contract=off: no fused multiply-add, so every fp32 step of the quantizer is
# one IEEE operation on every host (GCC contracts by default on aarch64).
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
