"""Builds libfa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each translation unit compiles in parallel; the objects link into one shared
library with the CUDA runtime linked statically, so the library does not
depend on the runtime version that PyTorch brings.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libfa.so")

SOURCES = ["fa_api.cu", "fa_simt.cu", "fa_tc_fwd.cu", "fa_tc_bwd.cu", "fa_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags(debug: bool):
    f = ARCH + ["-std=c++20", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if debug:
        f += ["-DFA_DEBUG=1"]
    return f


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, debug: bool = False, ptxas_v: bool = False) -> str:
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "fa.h"))
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) > max(os.path.getmtime(p) for p in deps)):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    objs = [os.path.join(BUILD_DIR, os.path.basename(s).replace(".cu", ".o")) for s in srcs]
    extra = ["-Xptxas", "-v"] if ptxas_v else []

    def one(pair):
        s, o = pair
        return _run([cc, *_flags(debug), *extra, "-c", s, "-o", o])

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        logs = list(ex.map(one, zip(srcs, objs)))
    tmp = LIB_PATH + ".tmp"
    _run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static", "-Xcompiler", "-fPIC"])
    os.replace(tmp, LIB_PATH)
    if verbose or ptxas_v:
        sys.stdout.write("".join(logs))
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv)
    print(LIB_PATH)
