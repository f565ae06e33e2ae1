"""Build step for the CPU oracle (test infrastructure): gcc -> liboracle.so.

Plain C11 with pthreads; no CUDA, nothing shared with the GPU library.
"""
from __future__ import annotations

import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")


def library_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def stale() -> bool:
    lib = library_path()
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(_SRC)


def build(verbose: bool = False) -> str:
    out = library_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra", "-Werror",
           "-o", tmp, _SRC, "-lpthread"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)   # atomic: concurrent test processes never see a half-written file
    return out


if __name__ == "__main__":
    print(build(verbose=True))
