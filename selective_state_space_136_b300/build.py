"""Build the ss_scan CUDA library (and the ALU probe) in-tree for sm_103a.

    python -m selective_state_space_136_b300.build [--force]

Each .cu file compiles to an object under _build/ (in parallel), then the
objects link into selective_state_space_136_b300/libss_scan.so with the CUDA
runtime linked statically. Only files whose sources or headers changed are
rebuilt.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(ROOT, "_build")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "-I" + os.path.join(ROOT, "include")]

LIBS = {
    # library name -> sources
    "libss_scan.so": ["ss_api.cu", "ss_simple.cu", "ss_update.cu", "ss_rows.cu",
                      "ss_seq.cu", "ss_pair.cu", "ss_noalloc.cu", "ss_conv.cu", "ss_bwd.cu", "ss_ssd.cu", "ss_ssd_tc.cu"],
    "libss_probe.so": ["alu_probe.cu"],
}


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, force):
    obj = os.path.join(OBJ, os.path.basename(src)[:-3] + ".o")
    if force or _stale(obj, [src] + _headers()):
        tmp = obj + ".tmp"
        subprocess.check_call([NVCC] + FLAGS + ["-c", src, "-o", tmp])
        os.replace(tmp, obj)
    return obj


def build(force: bool = False, verbose: bool = False) -> dict:
    os.makedirs(OBJ, exist_ok=True)
    out = {}
    jobs = []
    for lib, srcs in LIBS.items():
        srcs = [os.path.join(CSRC, s) for s in srcs if os.path.exists(os.path.join(CSRC, s))]
        jobs.append((lib, srcs))
    all_srcs = [s for _, srcs in jobs for s in srcs]
    with ThreadPoolExecutor(max(1, min(len(all_srcs), os.cpu_count() or 1))) as ex:
        objs = dict(zip(all_srcs, ex.map(lambda s: _compile(s, force), all_srcs)))
    for lib, srcs in jobs:
        target = os.path.join(PKG, lib)
        o = [objs[s] for s in srcs]
        if force or _stale(target, o):
            tmp = target + ".tmp"
            subprocess.check_call([NVCC] + ARCH + ["-shared", "-o", tmp] + o)
            os.replace(tmp, target)
        out[lib] = target
        if verbose:
            print("built", target)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
