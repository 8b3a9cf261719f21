"""Build the CPU oracle (plain C) into oracle/libep_oracle.so with gcc.

Test infrastructure: the oracle is compiled so the test suite, the smoke check
and the benchmark's CPU-baseline leg can call it; the product library never
links or loads it.  A second build with -fopenmp (oracle/libep_oracle_omp.so)
splits the oracle's token loops over the host's cores for the benchmark's
all-cores baseline; where the compiler has no OpenMP it is skipped.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ep_oracle.c")
LIB = os.path.join(HERE, "libep_oracle.so")
LIB_OMP = os.path.join(HERE, "libep_oracle_omp.so")
FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]


def _compile(out, extra):
    tmp = out + ".tmp.%d" % os.getpid()
    subprocess.run(["gcc"] + FLAGS + extra + ["-o", tmp, SRC, "-lm"], check=True)
    os.replace(tmp, out)


def _fresh(path):
    return os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if force or not _fresh(LIB):
        _compile(LIB, [])
    return LIB


def build_omp(force: bool = False):
    """The OpenMP build's path, or None when the compiler cannot build it."""
    if force or not _fresh(LIB_OMP):
        try:
            _compile(LIB_OMP, ["-fopenmp"])
        except (subprocess.CalledProcessError, OSError):
            return None
    return LIB_OMP


if __name__ == "__main__":
    print(build(force=True))
    print(build_omp(force=True))
