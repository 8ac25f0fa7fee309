"""Compiles the CPU oracle (test infrastructure) into oracle/libkivi_oracle.so.

Flags: -O2 -ffp-contract=off and no fast-math, so that each fp32 operation in
the quantizer is one IEEE operation rounded to nearest-even on every host
(x86-64 and aarch64 alike; GCC would otherwise fuse multiply-adds on aarch64).
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kivi_oracle.cpp")
HDR = os.path.join(HERE, "kivi_oracle.h")
LIB_PATH = os.path.join(HERE, "libkivi_oracle.so")


def build(force: bool = False) -> str:
    """Builds the oracle library if it is missing or older than its sources."""
    if not force and os.path.exists(LIB_PATH):
        lib_t = os.path.getmtime(LIB_PATH)
        if lib_t >= os.path.getmtime(SRC) and lib_t >= os.path.getmtime(HDR):
            return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-Wall", "-Wextra", "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True))
