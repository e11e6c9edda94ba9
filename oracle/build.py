"""Builds the fp64 CPU oracle (test infrastructure) into oracle/lib/."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "flint_moe_ref.c")
LIB_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIB_DIR, "libflint_oracle.so")


def compile_to(src: str, out: str) -> str:
    """gcc build of one oracle source file into a shared library."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall",
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc if the library is missing or stale."""
    os.makedirs(LIB_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    compile_to(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
