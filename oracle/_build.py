"""Compiles the CPU oracle (oracle.c) into a shared library next to it.

Test infrastructure: called by the oracle package on first import and by the
repository's build entry point.  Plain gcc, no CUDA, no vectorised math flags:
``-ffp-contract=off`` keeps every float add a separate IEEE-754 binary32 add
(GCC's default on aarch64 would otherwise fuse multiply-adds).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "_build", "liborc.so")

CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra", "-Werror"]


def build(force: bool = False) -> str:
    """Builds ``_build/liborc.so`` if it is missing or older than oracle.c."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [os.environ.get("CC", "gcc"), *CFLAGS, SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
