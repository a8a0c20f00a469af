"""Compile the CPU oracle (oracle.c) into oracle/liboracle.so with gcc.

Test infrastructure only: the library this makes is loaded by the tests, by
the package smoke check and by the CPU-baseline leg of the benchmark, never by
the product path.  Flags keep the arithmetic identical on x86_64 and aarch64
(no fused multiply-add contraction, no -march).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT = os.path.join(HERE, "liboracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False, verbose: bool = False) -> str:
    """Build liboracle.so if it is missing or older than oracle.c; return its path."""
    if (not force and os.path.exists(OUT)
            and os.path.getmtime(OUT) >= os.path.getmtime(SRC)):
        return OUT
    tmp = OUT + ".tmp.%d" % os.getpid()
    last = None
    for omp in (["-fopenmp"], []):
        cmd = ["gcc", *BASE_FLAGS, *omp, SRC, "-o", tmp, "-lm"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        proc = subprocess.run(cmd, capture_output=True, text=True)
        if proc.returncode == 0:
            os.replace(tmp, OUT)
            return OUT
        last = proc.stderr
    raise RuntimeError("oracle build failed:\n" + (last or ""))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
