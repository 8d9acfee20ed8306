"""Compile the oracle's plain C source into ``oracle/liboracle.so``.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Built with gcc and
OpenMP, IEEE arithmetic kept strict: no fast-math, no FMA contraction.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
          "-Wall", "-shared", "-fPIC"]


def build(src: str = SRC, out: str = LIB, extra=()) -> str:
    """Compile ``src`` to the shared library ``out`` (rebuilt when stale)."""
    if (os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)
            and not extra):
        return out
    cmd = ["gcc", *CFLAGS, *extra, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(*sys.argv[1:2]))
