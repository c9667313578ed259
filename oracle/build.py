"""Compile the plain-C oracle into ``oracle/_build/liboracle.so`` with gcc.

Test infrastructure: the oracle is the independent checker of the CUDA library.
It is built with OpenMP over requests when the compiler supports it (the result
of every request is computed by one thread in a fixed order, so the output does
not depend on the thread count).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dspark_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", SRC, "-lm"]
    tmp = LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-o", tmp],
                       check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
