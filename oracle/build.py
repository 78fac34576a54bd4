"""Builds the CPU oracle (``libstmat_oracle.so``) with the host C compiler.

Test infrastructure only: the oracle is built here and loaded by the tests,
the smoke check and the benchmark's CPU-baseline leg; the product library
never links it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "stmat_oracle.c")
LIB = os.path.join(HERE, "libstmat_oracle.so")

# -ffp-contract=off and no fast-math: the scaled-fp8 product must stay one
# IEEE binary32 multiply, and NaN tests must not be folded away.
CFLAGS = ["-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    """Compiles the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cc = os.environ.get("CC", "gcc")
    subprocess.run([cc, *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
