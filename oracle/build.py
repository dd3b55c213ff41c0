"""Build the C++ oracle (test infrastructure) into oracle/_build/libecho_oracle.so.

    python -m oracle.build [--force]

Plain g++ (C++17, -O2, no fused multiply-add, OpenMP for independent token scores).
It shares no source, header or flag set with the CUDA library's build.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "echo_oracle.cpp")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libecho_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-fopenmp"]


def compiler() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("no C++ compiler (g++) found: the oracle needs one")


def stale() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(SRC) > os.path.getmtime(LIB)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    tmp = f"{LIB}.{os.getpid()}.tmp"
    cmd = [compiler(), *FLAGS, SRC, "-o", tmp]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)                # atomic: concurrent builders never see a partial file
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
