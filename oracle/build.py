"""Build the CPU oracle shared library with gcc (test infrastructure)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "uq_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "libuq_oracle.so")

# Plain IEEE arithmetic: no fast-math and no fused multiply-add contraction,
# so the fp32 rotation and fp64 sums round as written in the source.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
          "-ffp-contract=off", "-pthread"]


def build_oracle(force: bool = False) -> str:
    """Compile uq_oracle.c into _build/libuq_oracle.so if it is out of date."""
    if (not force and os.path.exists(OUT)
            and os.path.getmtime(OUT) >= os.path.getmtime(SRC)):
        return OUT
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = OUT + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build_oracle(force=True))
