"""Compile the C oracle (plain gcc, no CUDA). Test infrastructure only.

Two builds of the one source ``attention_oracle.c``:

- ``liboracle.so``: the parity oracle, fp64 accumulation, one thread, -O2.
- ``liboracle_fp32omp.so``: the timed CPU baseline, the same loops with fp32
  accumulation (-DORC_ACC_FLOAT), -O3 and OpenMP over the selected rows.

Built on whichever machine runs the tests, so both use portable flags (no
-march / -mcpu, no architecture-specific code): the benchmark host is an Arm
box, this build host an x86 one.
"""
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "attention_oracle.c")
LIB = os.path.join(_HERE, "liboracle.so")
LIB_FAST = os.path.join(_HERE, "liboracle_fp32omp.so")


def _fresh(lib):
    return os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(SRC)


def _cc(out, flags):
    tmp = out + ".%d.tmp" % os.getpid()
    subprocess.run(["gcc"] + flags + ["-std=c99", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"],
                   check=True, capture_output=True)
    os.replace(tmp, out)


def build_oracle(force: bool = False) -> str:
    """The fp64 parity oracle (the one the tests compare against)."""
    if force or not _fresh(LIB):
        _cc(LIB, ["-O2"])
    return LIB


def build_oracle_fp32omp(force: bool = False) -> str:
    """The timed baseline build: fp32 accumulation, -O3, OpenMP (if the
    compiler has it; else one thread, which ``oracle_threads()`` reports)."""
    if force or not _fresh(LIB_FAST):
        try:
            _cc(LIB_FAST, ["-O3", "-fopenmp", "-DORC_ACC_FLOAT"])
        except subprocess.CalledProcessError:
            _cc(LIB_FAST, ["-O3", "-DORC_ACC_FLOAT"])
    return LIB_FAST


def build_all(force: bool = False):
    return build_oracle(force), build_oracle_fp32omp(force)


if __name__ == "__main__":
    print(build_all(force=True))
