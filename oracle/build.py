"""Compile the CPU oracle (plain C++17, g++) into oracle/liboracle.so.

Test infrastructure: the oracle is built so that it can check the CUDA path; the
product never loads it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if force or not up_to_date():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
