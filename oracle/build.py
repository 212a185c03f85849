"""Compile the C oracle (``oracle.c``) into ``liboracle.so`` with gcc.

Test infrastructure only: called by the test suite, by the build entry point
(building the checker is not using it) and by the benchmark's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    """Build ``liboracle.so`` next to this file if missing or stale; return its path."""
    stale = (not os.path.exists(LIBRARY)) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)
    if force or stale:
        tmp = LIBRARY + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c99", "-Wall", "-Wextra", "-shared", "-fPIC",
               "-o", tmp, SOURCE, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build_oracle(force=True))
