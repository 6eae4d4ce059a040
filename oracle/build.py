"""Build the fp64 CPU oracle (test infrastructure) into oracle/liboracle.so.

The oracle is plain C compiled with gcc and OpenMP, with no fast-math and no
fused multiply-add contraction, so each operation rounds as written.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(src=SRC, out=LIB, extra_flags=()):
    """Compile `src` into the shared library `out`; rebuild only when stale."""
    if (os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)
            and not extra_flags):
        return out
    cmd = ["gcc", *CFLAGS, *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build())
    sys.exit(0)
