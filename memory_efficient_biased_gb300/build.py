"""Build libevo_attn.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

    python -m memory_efficient_biased_gb300.build [--force] [-j N]

Each translation unit under csrc/ compiles in parallel to an object under
_build/, then nvcc links the shared library into memory_efficient_biased_gb300/_lib/.
The throughput microbenchmarks under csrc/micro/ (run by `bench.py --micro`)
link into a library of their own, libevo_micro.so.  Objects are rebuilt only
when a source or header is newer than them.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libevo_attn.so")
MICRO_LIB = os.path.join(LIBDIR, "libevo_micro.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libevo_attn.so")
    return p


def sources(sub: str = ""):
    d = os.path.join(CSRC, sub)
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _newest(paths):
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def build(force: bool = False, jobs: int = 8, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    hdr_time = _newest(headers())
    cmds = []
    libs = {LIB: [], MICRO_LIB: []}
    for lib, sub in ((LIB, ""), (MICRO_LIB, "micro")):
        for src in sources(sub):
            obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
            libs[lib].append(obj)
            if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_time):
                cmds.append([nvcc(), *ARCH, *CFLAGS, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}")

    with ThreadPoolExecutor(max_workers=max(1, jobs)) as ex:
        list(ex.map(run, cmds))
    for lib, objs in libs.items():
        if cmds or not os.path.exists(lib) or os.path.getmtime(lib) < _newest(objs):
            link = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", lib, *objs]
            r = subprocess.run(link, capture_output=True, text=True)
            if r.returncode:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-j", type=int, default=8)
    ap.add_argument("-v", action="store_true")
    a = ap.parse_args()
    print(build(a.force, a.j, a.v))
