"""In-tree build of libsoftmax.so for sm_103a (nvcc, no cmake).

Each translation unit is compiled to an object in parallel, then linked into
row_wise_softmax_gb300/libsoftmax.so.  A rebuild happens only when a source or
header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsoftmax.so")

SOURCES = ["softmax_abi.cu", "plan.cpp", "warp_rows.cu", "tile_rows.cu", "row_slices.cu",
           "row_slices_options.cu", "twopass.cu", "stream_rows.cu", "backward_rows.cu",
           "columns.cu", "columns_stream.cu", "attention_mma.cu", "attention_tc.cu"]
# Sources that include another source file.
INCLUDED = {"row_slices_options.cu": ["row_slices.cu"]}
HEADERS = [os.path.join(CSRC, h) for h in ("common.cuh", "kernels.h", "cluster_ring.cuh",
                                            "tensor_map.h", "attention_pp.h")] + [
    os.path.join(INCLUDE, "softmax.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-I", INCLUDE, "-I", CSRC, *ARCH]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libsoftmax")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, verbose: bool) -> str:
    cmd = [nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    """Build libsoftmax.so if any source changed; returns its path."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not _stale(LIB, srcs + HEADERS + [os.path.abspath(__file__)]):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    objs = [os.path.join(BUILD, os.path.basename(s) + ".o") for s in srcs]
    deps = lambda s: ([s] + [os.path.join(CSRC, d) for d in INCLUDED.get(os.path.basename(s), [])]
                      + HEADERS + [os.path.abspath(__file__)])
    todo = [(s, o) for s, o in zip(srcs, objs) if force or verbose or _stale(o, deps(s))]
    logs = []
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo) or 1, os.cpu_count() or 4)) as ex:
        for log in ex.map(lambda so: _compile(so[0], so[1], verbose), todo):
            logs.append(log)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), "-shared", *ARCH, "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    if verbose:
        print("".join(logs))
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
