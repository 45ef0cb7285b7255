"""Compile the C oracle into oracle/libmoe_oracle.so (plain gcc, OpenMP).

-ffp-contract=off keeps every multiply and add a separately rounded IEEE
operation, so the compiler cannot fuse or reorder the oracle's arithmetic.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "libmoe_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-Wall", "-Wextra", "-shared",
           "-fPIC", "-o", LIB, SRC, "-lm"]
    subprocess.check_call(cmd)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
