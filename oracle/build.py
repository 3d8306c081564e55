"""Compile the fp64 CPU oracle (test infrastructure) into a shared library.

Plain gcc, no CUDA: the oracle shares nothing with the GPU library.
Usable as ``python -m oracle.build`` or through ``build_oracle()``.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libattn_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Build ``oracle/_build/libattn_oracle.so`` if it is missing or stale."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    # -O2 without fast-math: IEEE double arithmetic in source order.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
