"""Builds the oracle's shared library with the host C compiler.

Test infrastructure: the CUDA library does not depend on this file.
Plain ``-O2`` without fast-math, so that IEEE double semantics hold.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = [os.path.join(HERE, "csa_oracle.c"), os.path.join(HERE, "csa_oracle_backward.c")]
LIB_PATH = os.path.join(HERE, "libcsa_oracle.so")


def build_oracle(verbose: bool = False) -> str:
    cc = os.environ.get("CC", "gcc")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-o", tmp] + SOURCES + ["-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_oracle(verbose=True))
