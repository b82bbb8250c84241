"""Compile the C oracle into ``oracle/liboracle.so`` (test infrastructure only).

Plain gcc, no machine-specific flags, so the same source gives the same
results on x86-64 and aarch64 hosts.  ``-ffp-contract=off`` keeps every fp64
multiply and add separately rounded, exactly as written in ``oracle.c``.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
HDR = os.path.join(HERE, "oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False) -> str:
    if force or is_stale():
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", "-Wall", SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
