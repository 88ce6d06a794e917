"""Builds the oracle's shared library (oracle/libmoe_oracle.so) with the host C compiler.

The oracle is test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline load it. -ffp-contract=off keeps multiply-adds unfused so x86 and Arm hosts agree.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "libmoe_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-Wall", "-Wextra"]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the oracle if the library is missing or older than its sources; returns its path."""
    srcs = [SRC, os.path.join(HERE, "moe_oracle.h")]
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(s) for s in srcs):
            return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc, *CFLAGS, SRC, "-o", tmp, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
