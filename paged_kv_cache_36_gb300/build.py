"""Builds libpkv.so in-tree for sm_103a.

CUDA sources are compiled by nvcc for `-gencode arch=compute_103a,code=sm_103a`
and host C++ sources by the host compiler, in parallel; the objects are linked
into paged_kv_cache_36_gb300/libpkv.so.  A rebuild happens only when a source,
header or flag changed (a stamp file in _build/ records the inputs' hash).

Run `python -m paged_kv_cache_36_gb300.build` or call build().
"""

from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-I", CSRC]


def _cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _stamp(cuda: str) -> str:
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["../../include/pkv.h"]
    for f in files:
        path = os.path.normpath(os.path.join(CSRC, f))
        if os.path.isfile(path):
            h.update(f.encode())
            with open(path, "rb") as fh:
                h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + CXX_FLAGS + [cuda, os.uname().machine]).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of libpkv.so."""
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    cxx = os.environ.get("CXX", "g++")
    os.makedirs(BUILD, exist_ok=True)
    stamp_file = os.path.join(BUILD, "stamp")
    stamp = _stamp(cuda)
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB
    cu, cpp = _sources()
    jobs = []
    for f in cu:
        obj = os.path.join(BUILD, f + ".o")
        jobs.append([nvcc] + NVCC_FLAGS + ["-c", os.path.join(CSRC, f), "-o", obj])
    for f in cpp:
        obj = os.path.join(BUILD, f + ".o")
        jobs.append([cxx] + CXX_FLAGS + ["-c", os.path.join(CSRC, f), "-o", obj])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        for msg in ex.map(run, jobs):
            if verbose and msg:
                print(msg)
    objs = [os.path.join(BUILD, f + ".o") for f in cu + cpp]
    tmp = LIB + ".tmp"
    run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs +
        ["-L", os.path.join(cuda, "lib64"), "-lcudart"])
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
