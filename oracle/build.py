"""Compile the C oracle into ``oracle/liboracle.so`` (plain gcc, no CUDA).

Test infrastructure only. Built on whichever machine runs the tests, so it uses
portable flags (no -march) and no architecture-specific code.
"""
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "attention_oracle.c")
LIB = os.path.join(_HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
