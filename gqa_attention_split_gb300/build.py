"""Builds libgqa_attn.so in-tree with nvcc for sm_103a (no cmake, no torch).

Every translation unit compiles in parallel to ``_build/`` at the repository
root; the shared library lands next to this file. A rebuild happens only when
a source or header is newer than the library.

    python -m gqa_attention_split_gb300.build [--force] [--verbose] [--debug]
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgqa_attn.so")
DEBUG_LIB = os.path.join(PKG, "libgqa_attn_debug.so")

SOURCES = ["plan.cpp", "runtime.cu", "decode.cu", "prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Hidden visibility: only the C ABI (GQA_API in include/gqa_attn.h) is exported,
# so two builds loaded in one process (the product and the -DGQA_DEBUG library)
# share no C++ symbols, template statics included.
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgqa_attn.so")


def _newest_input() -> float:
    t = 0.0
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            t = max(t, os.path.getmtime(os.path.join(d, f)))
    return max(t, os.path.getmtime(__file__))


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          debug: bool = False) -> str:
    """Builds the library; ``debug=True`` builds the -DGQA_DEBUG variant
    (``libgqa_attn_debug.so``, with the prefill tile counters) instead.
    Returns the library's path."""
    lib = DEBUG_LIB if debug else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    nvcc = _nvcc()
    out_dir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(out_dir, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src + ".o")
        extra = os.environ.get("GQA_EXTRA_NVCC_FLAGS", "").split()
        if debug:
            extra.append("-DGQA_DEBUG")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose and src.endswith(".cu"):
            cmd.insert(1, "-Xptxas=-v")
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if (verbose or ptxas_verbose) and r.stderr:
            print(r.stderr, file=sys.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the -DGQA_DEBUG variant")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose, debug=a.debug))
