"""Build the CPU oracle library (test infrastructure only).

Compiles ``bloom_oracle.c`` with the host C compiler into ``liborc.so`` beside
this file.  No fast-math: the oracle keeps IEEE double semantics and the
summation order written in the source.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bloom_oracle.c")
LIB = os.path.join(HERE, "liborc.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
        os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "bloom_oracle.h"))
    ):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc, "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
