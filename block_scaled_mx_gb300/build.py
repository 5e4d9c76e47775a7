"""Build libmxmoe.so in-tree: every CUDA translation unit compiled in parallel
for sm_103a only, then linked into one shared library next to this file.

Rebuilds are keyed on a stamp: a hash of every source and header, the compile
flags and the nvcc version.  The stamp is compiled into the library
(``mx_build_stamp()``) and written beside it; a library whose stamp differs from
the current sources is rebuilt, whatever the file times say, so a library copied
from another machine or built from other sources is never used.
"""
from __future__ import annotations

import hashlib
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libmxmoe.so")
STAMP_FILE = LIB + ".stamp"
SOURCES = ["prep.cu", "gemm.cu", "router.cu", "api.cu", "noalloc.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]

# what the last build() call in this process did: {"stamp", "compiled", "lib"}
LAST_BUILD: dict = {}


def _inputs():
    headers = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh")))
    headers.append(os.path.join(ROOT, "include", "mxmoe.h"))
    return [os.path.join(CSRC, s) for s in SOURCES] + headers


def _nvcc_version() -> str:
    try:
        return subprocess.run([NVCC, "--version"], capture_output=True, text=True).stdout.strip()
    except OSError:
        return "nvcc unavailable"


def source_stamp(extra_flags=None) -> str:
    """16 hex digits of sha256 over the sources, headers, flags and nvcc version."""
    h = hashlib.sha256()
    for path in _inputs():
        h.update(os.path.relpath(path, ROOT).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(FLAGS + list(extra_flags or [])).encode())
    h.update(_nvcc_version().encode())
    return h.hexdigest()[:16]


def built_stamp() -> str | None:
    """The stamp written beside the library by the build that made it."""
    try:
        with open(STAMP_FILE) as f:
            return f.read().strip()
    except OSError:
        return None


def build(verbose: bool = False, extra_flags=None) -> str:
    stamp = source_stamp(extra_flags)
    if os.path.exists(LIB) and built_stamp() == stamp:
        LAST_BUILD.update(stamp=stamp, compiled=False, lib=LIB)
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    flags = FLAGS + list(extra_flags or []) + [f"-DMXMOE_BUILD_STAMP=\"{stamp}\""]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [NVCC, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP_FILE, "w") as f:
        f.write(stamp + "\n")
    sys.stderr.write(f"libmxmoe.so: compiled {len(SOURCES)} CUDA sources with nvcc for sm_103a, stamp {stamp}\n")
    LAST_BUILD.update(stamp=stamp, compiled=True, lib=LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else None))
