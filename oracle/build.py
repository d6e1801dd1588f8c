"""Builds the CPU oracle (test infrastructure) into oracle/_build/liboracle.so.

The oracle is plain C, compiled with contraction and fast-math off so that
every product and every sum is rounded on its own (no fused multiply-add).
It shares no code with the CUDA library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "repops_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing", "-fPIC", "-shared", "-Wall"]
LDLIBS = ["-lm"]


def build(force: bool = False) -> str:
    """Compiles the oracle if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [os.environ.get("CC", "gcc")] + CFLAGS + ["-o", tmp, SRC] + LDLIBS
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
