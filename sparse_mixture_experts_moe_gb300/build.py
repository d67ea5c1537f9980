"""Builds the layer's CUDA library (libmoe.so) and the input generator's device fill
(inputgen/libinputgen.so) in-tree for sm_103a with nvcc.

Each .cu file compiles to an object in parallel; the objects link into one shared
library with the CUDA runtime linked statically, so loading the library needs no
GPU and no CUDA driver (its entry points only touch the driver when called).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]

LIB_SOURCES = ["api.cu", "router.cu", "router_tc.cu", "router_small.cu", "dispatch.cu", "dispatch_noalloc.cu",
               "ffn_simt.cu", "ffn_stream.cu", "ffn_tc.cu", "ffn_tc2.cu", "combine.cu", "graph.cu", "quant.cu",
               "ffn_tct.cu"]
LIB_PATH = os.path.join(PKG, "libmoe.so")
INPUTGEN_SRC = os.path.join(ROOT, "inputgen", "fill.cu")
INPUTGEN_PATH = os.path.join(ROOT, "inputgen", "libinputgen.so")


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(verbose: bool = False, ptxas_info: bool = False) -> None:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for src in LIB_SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        jobs.append(([nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj], obj))
    ig_obj = os.path.join(BUILD, "inputgen_fill.o")
    jobs.append(([nvcc, *ARCH, *FLAGS, "-c", INPUTGEN_SRC, "-o", ig_obj], ig_obj))
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        outs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose or ptxas_info:
        for (cmd, _), out in zip(jobs, outs):
            if out.strip():
                print(out, file=sys.stderr)
    lib_objs = [j[1] for j in jobs[:-1]]
    _run([nvcc, *ARCH, "-shared", "-o", LIB_PATH, *lib_objs])
    _run([nvcc, *ARCH, "-shared", "-o", INPUTGEN_PATH, ig_obj])


if __name__ == "__main__":
    build(verbose=True, ptxas_info="--ptxas" in sys.argv)
