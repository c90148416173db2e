"""Build the CPU oracle (test infrastructure) into oracle/_lib/liboracle.so.

Plain gcc, -O2, no fast-math and no fused multiply-adds (-ffp-contract=off), so the
f32 arithmetic is the source's, in the source's order, on x86 and on Arm alike.
OpenMP only splits independent rows/heads.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rq_oracle.c")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wno-unknown-pragmas",
           SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
