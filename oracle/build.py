"""Compile the CPU oracle (oracle.c) into liboracle.so beside this file.

TEST INFRASTRUCTURE ONLY: the oracle is the checker for the CUDA library, not
part of it.  Plain gcc, no fast-math, no FMA contraction, so every float
expression in oracle.c is one IEEE operation.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = [
    "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
    "-ffp-contract=off", "-fno-fast-math", "-fno-finite-math-only",
    "-Wall", "-Wextra", "-Wno-unused-parameter",
]


def _stale(lib: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(SRC)


def build(force: bool = False, mutant: int = 0) -> str:
    """Build liboracle.so if missing or older than oracle.c; return its path.

    ``mutant`` > 0 builds a copy with one deliberate mistake planted (see the
    ORACLE_MUTANT blocks in oracle.c) under _mutants/; the test-suite uses
    those copies to show that its pins catch such mistakes.
    """
    if mutant:
        d = os.path.join(HERE, "_mutants")
        os.makedirs(d, exist_ok=True)
        lib = os.path.join(d, "liboracle_mut%d.so" % mutant)
    else:
        lib = LIB
    if force or _stale(lib):
        tmp = lib + ".tmp%d" % os.getpid()
        extra = ["-DORACLE_MUTANT=%d" % mutant] + (["-w"] if mutant else [])
        cmd = [os.environ.get("CC", "gcc")] + CFLAGS + extra + [SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
