"""Build step for the CPU oracle (test infrastructure only).

Compiles ``sc_oracle.cpp`` with g++ (OpenMP when available) into
``liboracle.so`` next to this file.  Nothing here is used by the CUDA
library; the test suite, the smoke check and the benchmark's CPU-baseline leg
are the only callers.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sc_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, src: str = SRC, lib: str = LIB) -> str:
    """Compile `src` into the shared library `lib` (default: the oracle)."""
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) >= os.path.getmtime(src)):
        return lib
    tmp = lib + ".tmp%d" % os.getpid()
    base = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", src, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)  # no OpenMP: single-threaded oracle
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
