"""Compile libtreeattn.so in-tree with nvcc for sm_103a.

Every translation unit is compiled in parallel; the shared library links the
CUDA runtime statically, so loading it needs no CUDA library path. A stamp of
the sources' contents and flags decides whether a rebuild is needed.
"""
from __future__ import annotations

import fcntl
import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtreeattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr", f"-I{INCLUDE}"]
CXX_FLAGS = ["-x", "c++", "-std=c++17", "-O2", "-fPIC"]  # host sources, driven through nvcc


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    srcs = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))
    deps = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh")))
    deps.append(os.path.join(INCLUDE, "treeattn.h"))
    return srcs, deps


def _stamp(srcs, deps) -> str:
    h = hashlib.sha256()
    for path in srcs + deps:
        h.update(path.encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + CXX_FLAGS).encode())
    return h.hexdigest()


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Build (if stale) and return the path of libtreeattn.so."""
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        srcs, deps = _sources()
        stamp = _stamp(srcs, deps)
        stamp_file = os.path.join(BUILD, "stamp")
        if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
            with open(stamp_file) as f:
                if f.read().strip() == stamp:
                    return LIB
        nvcc = _nvcc()
        jobs = []
        objs = []
        for src in srcs:
            obj = os.path.join(BUILD, os.path.basename(src) + ".o")
            objs.append(obj)
            if src.endswith(".cu"):
                cmd = [nvcc] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + ["-c", src, "-o", obj]
            else:  # host C++: nvcc drives the host compiler with the CUDA include path
                cmd = [nvcc, "-x", "c++", "-std=c++17", "-O2", "-Xcompiler", "-fPIC",
                       f"-I{INCLUDE}", "-c", src, "-o", obj]
            jobs.append(cmd)
        with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            logs = list(ex.map(_run, jobs))
        if verbose:
            for log in logs:
                if log.strip():
                    print(log)
        tmp = LIB + ".tmp"
        _run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-ldl", "-lrt", "-lpthread"])
        os.replace(tmp, LIB)
        with open(stamp_file, "w") as f:
            f.write(stamp)
        return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
