"""Compile the CPU oracle (oracle.c) into liboracle.so with gcc.

Test infrastructure: building the checker is not using it. Run as `python -m oracle.build` or
call `build()`.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")


def build(source: str = SOURCE, output: str = LIBRARY, extra_flags=(), quiet: bool = False) -> str:
    """Compile `source` to the shared library `output` (fp64, -O2, OpenMP) and return its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", *extra_flags, source, "-o", output, "-lm"]
    if not quiet:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    return output


def needs_build(source: str = SOURCE, output: str = LIBRARY) -> bool:
    return not os.path.exists(output) or os.path.getmtime(output) < os.path.getmtime(source)


if __name__ == "__main__":
    build()
