"""Builds the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain g++ with -ffp-contract=off so that no multiply-add is contracted; the
oracle's binary32 steps are then single IEEE operations, as its header states.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.cpp")
HDR = os.path.join(HERE, "oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", "-Wall", "-o", tmp, SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
