"""Builds the CPU oracle (test infrastructure) into oracle/libgs2d_oracle.so.

Plain gcc, no CUDA.  -ffp-contract=off keeps the FP32 touch decision's
products and sums separately rounded, as the oracle's source requires.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gs2d_oracle.c")
LIB = os.path.join(HERE, "libgs2d_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


# The multi-threaded timing driver: the same source compiled with OpenMP
# around its per-pixel functions (gs2d_oracle_omp.c includes gs2d_oracle.c).
SRC_OMP = os.path.join(HERE, "gs2d_oracle_omp.c")
LIB_OMP = os.path.join(HERE, "libgs2d_oracle_omp.so")


def build_omp(force: bool = False) -> str:
    t = os.path.getmtime(LIB_OMP) if os.path.exists(LIB_OMP) else -1.0
    if not force and t >= max(os.path.getmtime(SRC), os.path.getmtime(SRC_OMP)):
        return LIB_OMP
    tmp = LIB_OMP + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
           "-shared", "-Wall", "-Wextra", "-I", HERE, "-o", tmp, SRC_OMP, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_OMP)
    return LIB_OMP


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
    print(build_omp(force="--force" in sys.argv))
