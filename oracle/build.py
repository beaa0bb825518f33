"""Builds the CPU oracle (oracle.c, oracle_attn.c, oracle_fp8.c) into liboracle.so next to this file.

Test infrastructure: plain gcc, no CUDA.  ``-ffp-contract=off`` keeps the double
arithmetic free of fused multiply-adds so x86 and Arm hosts round identically.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["oracle.c", "oracle_core.inc", "oracle_attn.c", "oracle_fp8.c", "oracle.h"]
LIB = os.path.join(HERE, "liboracle.so")


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in SOURCES)


def compile_library(src_dir: str, out: str) -> str:
    """Compiles the oracle sources found in `src_dir` into the shared library `out`."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-o", tmp, os.path.join(src_dir, "oracle.c"), os.path.join(src_dir, "oracle_attn.c"),
           os.path.join(src_dir, "oracle_fp8.c"), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or needs_build():
        compile_library(HERE, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
