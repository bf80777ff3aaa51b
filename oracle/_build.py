"""Build step for the oracle's C part (``la_oracle.c`` -> ``liblaoracle.so``).

Test infrastructure only: it compiles the checker, it runs nothing. Plain gcc,
fp64, OpenMP, no fast-math (the summation order is the one written in the C).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "la_oracle.c")
LIB = os.path.join(HERE, "liblaoracle.so")


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99",
           "-fno-fast-math", "-ffp-contract=off", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
