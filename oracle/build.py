"""Build the CPU oracle shared library with gcc.

Test infrastructure: the library this builds is loaded only by the test suite,
the smoke check and bench.py's CPU baseline leg.  Output goes to
oracle/_build/liborc.so (git-ignored).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "w4a16_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liborc.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
          "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile liborc.so if it is missing or older than its source; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)  # atomic: concurrent builders never see a half-written file
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
