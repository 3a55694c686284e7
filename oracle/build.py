"""Compile the fp64 CPU oracle (``recurrence.c``) into ``liboracle.so``.

Test infrastructure only: the tests, the package smoke check and the bench's
CPU-baseline leg are the only users. Plain gcc, no GPU, no CUDA headers.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "recurrence.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
