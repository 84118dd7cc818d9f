"""Compile the oracle's C part (moe_oracle.c) into oracle/_build/liboracle.so with gcc.

Test infrastructure only (see oracle/__init__.py).  Plain portable C: the same source
builds on x86_64 and aarch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "liboracle.so")


def build() -> str:
    os.makedirs(os.path.dirname(LIB_PATH), exist_ok=True)
    src = os.path.join(HERE, "moe_oracle.c")
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, src])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build())
