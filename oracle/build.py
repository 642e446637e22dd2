"""Build the FP64 CPU oracle (test infrastructure only) with the system C compiler.

    python oracle/build.py

Writes ``oracle/liboracle.so`` next to the source.  ``-ffp-contract=off`` keeps
every product and sum of the oracle a separately rounded FP64 operation, as
the oracle's RoPE reading states.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-Wextra", "-Wno-unused-parameter",
           SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
