"""Compile the oracle's C source into a shared library next to it.

TEST INFRASTRUCTURE ONLY: the oracle checks the CUDA path and is never part
of it.  gcc with OpenMP when available, plain gcc otherwise.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wextra"]
    tmp = LIB + ".tmp.%d" % os.getpid()
    for extra in (["-fopenmp"], []):
        cmd = base + extra + [SRC, "-o", tmp, "-lm"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
        last = r.stderr
    raise RuntimeError("oracle build failed:\n" + last)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
