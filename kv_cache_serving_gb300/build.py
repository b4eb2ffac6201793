"""Builds libdsa.so (sm_103a) in-tree under kv_cache_serving_gb300/_build/.

Each .cu in csrc/ is compiled by nvcc in parallel, then linked into one shared
library with the CUDA runtime linked statically.  A stamp file holds a hash of
the sources and flags, so an unchanged tree is not rebuilt.

    python -m kv_cache_serving_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libdsa.so")
STAMP = os.path.join(BUILD, "libdsa.stamp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-ffp-contract=off", "-I", INCLUDE, "-I", CSRC]

_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsa")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _digest(extra_flags) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                h.update(f.encode())
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def build(force: bool = False, extra_flags=(), verbose: bool = False) -> str:
    """Compile (if needed) and return the path of libdsa.so."""
    with _lock:
        digest = _digest(extra_flags)
        if not force and os.path.exists(LIB) and os.path.exists(STAMP):
            with open(STAMP) as f:
                if f.read().strip() == digest:
                    return LIB
        os.makedirs(BUILD, exist_ok=True)
        cc = nvcc()
        objs = []

        def compile_one(src):
            obj = os.path.join(BUILD, src[:-3] + ".o")
            cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr, flush=True)
            return obj

        srcs = sources()
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
            objs = list(ex.map(compile_one, srcs))
        tmp = f"{LIB}.{os.getpid()}.tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        with open(STAMP, "w") as f:
            f.write(digest)
        return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
