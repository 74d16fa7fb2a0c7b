"""Compile the CPU oracle into ``oracle/_lib/liboracle.so`` (gcc, no GPU).

Test infrastructure only: the oracle is built with strict IEEE float semantics
(no fast-math, no FMA contraction) so that every rounding step is the one its
source states.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "liboracle.so")
SRC = os.path.join(HERE, "ep_oracle.cpp")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
           "-shared", "-Wall", "-Wextra", "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
