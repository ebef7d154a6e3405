"""Compile libpmha.so (the CUDA library behind include/pmha.h) in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel; the objects are linked
into graph_sparse_head_gb300/libpmha.so with the CUDA runtime linked
statically, so the library loads on a machine without a GPU driver (the
symbols can be inspected there; every compute call needs a GB300).
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpmha.so")
SOURCES = ["api.cu", "csr.cu", "gemm_simt.cu", "gemm_tc.cu", "edge_attn.cu", "edge_attn_f16.cu", "edge_attn_f32.cu", "edge_attn_ring.cu", "edge_attn_ring_out.cu",
           "dense_attn.cu", "backward.cu", "bwd_ring.cu", "noalloc.cu", "heavy.cu"]
HEADERS = [os.path.join(CSRC, "pmha_internal.h"), os.path.join(CSRC, "edge_stream.cuh"), os.path.join(CSRC, "edge_ring.cuh"), os.path.join(CSRC, "edge_out.cuh"), os.path.join(CSRC, "bwd_stream.cuh"),
           os.path.join(CSRC, "tc_util.cuh"),
           os.path.join(ROOT, "include", "pmha.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "-Xptxas", "-warn-spills", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpmha.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), build_dir: str = BUILD,
          out_lib: str = LIB) -> str:
    """Compile the sources (only those older than their output) and link the library."""
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + HEADERS):
            jobs.append([cc, *FLAGS, *extra_flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for out in ex.map(run, jobs):
                if verbose and out.strip():
                    print(out, file=sys.stderr)
    if force or jobs or _stale(out_lib, objs):
        tmp = out_lib + f".tmp{os.getpid()}"
        run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
        os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
