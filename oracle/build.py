"""Build step for the oracle's shared library (test infrastructure only).

The oracle is plain C compiled with gcc; it is built on whichever machine
runs the tests, because a library compiled on one architecture does not
load on another.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it and return the path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-Wall", "-Wno-unknown-pragmas"]
    tmp = LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: the oracle still builds, single-threaded
        subprocess.run(base + [SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
