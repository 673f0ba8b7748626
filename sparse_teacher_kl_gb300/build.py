"""Build libkdkl.so in-tree from csrc/*.cu for sm_103a with nvcc.

Each translation unit is compiled in parallel into ``_build/``, then linked
(static CUDA runtime) into ``sparse_teacher_kl_gb300/libkdkl.so``.  A hash of
the sources, headers and flags skips the rebuild when nothing changed.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import re
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkdkl.so")
BUILD_DEBUG = os.path.join(ROOT, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libkdkl_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _digest(extra) -> str:
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)) + ["../../include/kdkl.h"]:
        path = os.path.normpath(os.path.join(CSRC, f))
        with open(path, "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    h.update(" ".join(ARCH + CFLAGS + extra).encode())
    return h.hexdigest()


def _code_only(text: bytes) -> bytes:
    """Source text without comments and blank space, so that a digest follows the code."""
    t = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    t = re.sub(rb"//[^\n]*", b"", t)
    return b"\n".join(line.strip() for line in t.splitlines() if line.strip())


def source_digest(files=None) -> str:
    """Digest of CUDA sources, comments and blank space left out (not of build flags):
    identifies the kernels that an ncu capture was taken from.  ``files``: names under
    csrc/ to digest (default: all of them and the public header)."""
    h = hashlib.sha256()
    names = sorted(files) if files is not None else sorted(os.listdir(CSRC)) + ["../../include/kdkl.h"]
    for f in names:
        path = os.path.normpath(os.path.join(CSRC, f))
        with open(path, "rb") as fh:
            h.update(os.path.basename(path).encode())
            h.update(_code_only(fh.read()))
    return h.hexdigest()[:16]


def build_library(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    """Compile and link libkdkl.so (or, with ``debug``, the checked libkdkl_debug.so:
    KD_DEBUG, kernels check their computed indices and report a bad one through the
    workspace error word instead of accessing it).  Returns the library path."""
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DKD_DEBUG=1"] if debug else [])
    bdir = BUILD_DEBUG if debug else BUILD
    lib = LIB_DEBUG if debug else LIB
    os.makedirs(bdir, exist_ok=True)
    stamp = os.path.join(bdir, os.path.basename(lib) + ".stamp")
    digest = _digest(extra)
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib
    nvcc = _nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for obj, log in results:
            if log.strip():
                sys.stderr.write(f"--- {os.path.basename(obj)}\n{log}\n")
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib


if __name__ == "__main__":
    build_library(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv)
    print(LIB)
