"""Builds libfa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each translation unit compiles in parallel; the objects link into one shared
library with the CUDA runtime linked statically, so the library does not
depend on the runtime version that PyTorch brings.  The debug library
(libfa_debug.so, -DFA_DEBUG=1) is built beside it from the same sources.
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
# the same sources with FA_DEBUG: in-kernel bounds checks and tile-load counters
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "libfa_debug.so")

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


def _build_one(lib_path: str, build_dir: str, debug: bool, force: bool, ptxas_v: bool):
    """(compile commands, link command, path) of one library, or None when the library
    is newer than every source."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "fa.h"))
    deps.append(os.path.abspath(__file__))
    if (not force and os.path.exists(lib_path)
            and os.path.getmtime(lib_path) > max(os.path.getmtime(p) for p in deps)):
        return None
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_v else []
    objs = [os.path.join(build_dir, os.path.basename(s).replace(".cu", ".o")) for s in srcs]
    compiles = [[cc, *_flags(debug), *extra, "-c", s, "-o", o] for s, o in zip(srcs, objs)]
    link = [cc, *ARCH, "-shared", "-o", lib_path + ".tmp", *objs, "-cudart", "static", "-Xcompiler", "-fPIC"]
    return compiles, link, lib_path


def build(force: bool = False, verbose: bool = False, debug: bool = True, ptxas_v: bool = False) -> str:
    """Builds libfa.so and (unless debug is False) libfa_debug.so, every translation
    unit of both in parallel; returns the release library's path."""
    jobs = [j for j in (_build_one(LIB_PATH, BUILD_DIR, False, force, ptxas_v),
                        _build_one(DEBUG_LIB_PATH, DEBUG_BUILD_DIR, True, force, False) if debug else None) if j]
    if not jobs:
        return LIB_PATH
    compiles = [c for j in jobs for c in j[0]]
    with ThreadPoolExecutor(max_workers=len(compiles)) as ex:
        logs = list(ex.map(_run, compiles))
    for _, link, path in jobs:
        _run(link)
        os.replace(path + ".tmp", path)
    if verbose or ptxas_v:
        sys.stdout.write("".join(logs))
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv)
    print(LIB_PATH)
