"""Compile the scalar CPU oracle (test infrastructure) into liboracle_zero1.so.

Plain gcc, no CUDA.  ``-ffp-contract=off`` keeps every fp32 multiply and add
a separately rounded operation on both x86-64 and Arm.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "zero1_oracle.c")
LIB = os.path.join(HERE, "liboracle_zero1.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def needs_build() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build_oracle(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + ".tmp.%d" % os.getpid()
        subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
