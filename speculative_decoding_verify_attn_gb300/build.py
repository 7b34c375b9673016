"""Build libspecverify.so in-tree with nvcc for sm_103a (GB300).

    python -m speculative_decoding_verify_attn_gb300.build [--force] [--verbose]

The library is written next to this file under ``_lib/`` (git-ignored).  Translation units are
compiled in parallel by nvcc (``--threads 0``); only one ``-gencode`` target is built.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIBNAME = "libspecverify.so"
LIBPATH = os.path.join(LIBDIR, LIBNAME)

SOURCES = ["attn.cu", "attn_tc.cu", "attn_tc_pair.cu", "sample.cu", "sample_tree.cu", "lmhead.cu", "commit.cu",
           "api.cpp", "noalloc.cu", "launch_cache.cpp"]
HEADERS = ["common.cuh", "attn_common.cuh", "tcgen05.cuh", "ff.cuh", "attn_internal.h", "sample_internal.h",
           "commit_internal.h", "lmhead_internal.h", "launch_cache.h"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin/ on PATH)")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "spec_verify.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIBPATH):
        return False
    t = os.path.getmtime(LIBPATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIBPATH
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = LIBPATH + ".tmp"
    cmd = [
        nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
        "--threads", "0", "-I", INCLUDE, "-I", CSRC,
        "-Xptxas", "-warn-spills",
        "-o", tmp,
    ] + [os.path.join(CSRC, s) for s in SOURCES] + ["-lpthread", "-ldl", "-lrt"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout, r.stderr, file=sys.stderr)
    os.replace(tmp, LIBPATH)
    return LIBPATH


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(path)
