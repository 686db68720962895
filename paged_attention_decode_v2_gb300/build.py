"""Build ``libpa.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file is compiled in parallel into ``_build/``, then the
objects are linked into ``paged_attention_decode_v2_gb300/libpa.so``.  A file
is recompiled only when it or a header under ``csrc/`` or ``include/`` is
newer than its object.

Usage: ``python -m paged_attention_decode_v2_gb300.build [--force] [--verbose]``
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(INCLUDE, "*.h")))


def _flags(verbose: bool):
    f = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE,
         "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_header = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    exe = nvcc()
    flags = _flags(verbose)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        if (not force and os.path.exists(obj) and
                os.path.getmtime(obj) >= max(os.path.getmtime(src), newest_header)):
            return obj, ""
        tmp = obj + f".tmp{os.getpid()}"
        r = subprocess.run([exe, *flags, "-c", src, "-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        os.replace(tmp, obj)
        return obj, r.stderr

    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    objs = [o for o, _ in results]
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(map(os.path.getmtime, objs)):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([exe, "-shared", *ARCH, *objs, "-o", tmp, "-cudart", "static",
                            "-Xlinker", "-Bsymbolic", "-Xlinker", "--exclude-libs,ALL"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libpa.so failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/spill reports")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
