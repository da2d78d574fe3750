"""Compile the CPU oracle (plain C) into oracle/libvr_oracle.so.

Test infrastructure: building the checker is not using it. The flags keep the
arithmetic exactly IEEE: no fast-math, no floating-point contraction.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vr_oracle.c")
LIB = os.path.join(HERE, "libvr_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def compile_oracle(src=SRC, out=LIB, extra=()):
    """Compile `src` into the shared library `out` with gcc; returns `out`."""
    cmd = ["gcc", *CFLAGS, *extra, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force=False):
    """Build the oracle library unless it is newer than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_oracle()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
