"""Build libw4a16.so (the CUDA library behind include/w4a16.h) for sm_103a.

Each .cu under csrc/ is compiled by its own nvcc process (in parallel), then
linked with the static CUDA runtime into int4_weight_only_gemv_gb300/_lib/
(git-ignored).  ptxas statistics are kept in _lib/ptxas.txt; a GEMV kernel
that spills registers or uses a stack frame fails the build.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libw4a16.so")
# The checked build: the same sources with W4A16_CHECKED, whose kernels check
# their indexes and set W4A16_DEV_INDEX instead of making an out-of-range
# access (a stand-in for a memory checker; slower, for tests only).
CHECKED_DIR = os.path.join(OUT_DIR, "checked")
CHECKED_LIB = os.path.join(CHECKED_DIR, "libw4a16_checked.so")
SOURCES = ["api.cu", "gemv_m1.cu", "gemv_rows.cu", "gemv_mma.cu", "quant.cu", "attn_decode.cu", "q4k.cu"]
HEADERS = ["kernels.h", "ptx.cuh"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _inputs() -> list[str]:
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] +
            [os.path.join(INCLUDE, "w4a16.h"), os.path.abspath(__file__)])


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile(src: str, out_dir: str, extra: list[str]) -> tuple[str, str]:
    obj = os.path.join(out_dir, os.path.basename(src).replace(".cu", ".o"))
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def _check_spills(log: str) -> list[str]:
    bad, fn = [], None
    for line in log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            fn = m.group(1)
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores", line)
        if m and fn and "gemv" in fn and (int(m.group(1)) or int(m.group(2))):
            bad.append(f"{fn}: {line.strip()}")
    return bad


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile the library (or, checked=True, its index-checked build) if any
    source is newer than it; return its path."""
    out_dir, lib = (CHECKED_DIR, CHECKED_LIB) if checked else (OUT_DIR, LIB)
    extra = ["-DW4A16_CHECKED"] if checked else []
    os.makedirs(out_dir, exist_ok=True)
    if not force and not _stale(lib):
        return lib
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda src: _compile(src, out_dir, extra), SOURCES))
    log = "\n".join(r[1] for r in results)
    with open(os.path.join(out_dir, "ptxas.txt"), "w") as f:
        f.write(log)
    bad = [] if checked else _check_spills(log)
    if bad:
        raise RuntimeError("register spills / stack frames in GEMV kernels:\n" + "\n".join(bad))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *[r[0] for r in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(log)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
