"""Build libpagedkv.so (the C-ABI library) for sm_103a with nvcc, in-tree.

Run `python paged_kv_cache_496_b300/build.py` (as a script: importing the package would load the
library it is about to build). The library is written next to this file.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(HERE, "libpagedkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def inputs():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) +
                              glob.glob(os.path.join(CSRC, "*.h")) +
                              glob.glob(os.path.join(INCLUDE, "*.h")))


def needs_build() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(f) > t for f in inputs())


def build(verbose: bool = False, extra=()) -> str:
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
           "--expt-relaxed-constexpr", *extra, *sources(), "-o", LIBRARY]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    return LIBRARY


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
