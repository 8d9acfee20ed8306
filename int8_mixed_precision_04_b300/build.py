"""Build ``libbnbint8.so`` in-tree with nvcc for sm_103a.

The library is plain CUDA C++ behind the C ABI of ``include/bnb_int8.h``; it
is built with nvcc directly (no torch extension machinery) so that it has no
dependence on torch at all.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libbnbint8.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-Wall", f"-I{os.path.join(ROOT, 'include')}"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(out):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = glob.glob(os.path.join(CSRC, "*")) + [os.path.join(ROOT, "include", "bnb_int8.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile every CUDA source into the shared library (if stale)."""
    if not force and not _stale(LIB):
        return LIB
    cmd = [NVCC, *ARCH, *FLAGS]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    cmd += [*sources(), "-o", LIB + ".tmp"]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
