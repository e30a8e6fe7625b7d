"""Compile the oracle's C part (oracle/hqr.c -> oracle/libhqr.so) with gcc.

Test infrastructure: builds the checker, not the product.  Plain C, no
architecture-specific flags, so it builds the same on x86-64 and AArch64."""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hqr.c")
LIB = os.path.join(HERE, "libhqr.so")


def build() -> str:
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", LIB + ".tmp", SRC, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build())
