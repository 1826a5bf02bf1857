"""Compiles the C oracle (gdn_oracle.c) into liboracle_gdn.so beside it.

Test infrastructure only: the oracle is the independent checker that tests,
the smoke check and the benchmark's CPU-baseline leg compare against.  Plain
gcc, -O2 without fast-math so that IEEE fp64 semantics hold, OpenMP over the
independent (sequence, head) units.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
LIB = os.path.join(HERE, "liboracle_gdn.so")


def build(force: bool = False, src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Builds `src` into the shared library `out` and returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
