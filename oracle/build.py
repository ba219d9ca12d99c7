"""Compile the CPU oracle (``spec_oracle.c``) into ``libspecoracle.so``.

Test infrastructure only: the oracle is built so the tests, the smoke check
and the benchmark's CPU-baseline leg can load it.  Plain gcc, no CUDA.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spec_oracle.c")
LIB = os.path.join(HERE, "libspecoracle.so")


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", SRC, "-o", LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the same arithmetic, one thread.
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
