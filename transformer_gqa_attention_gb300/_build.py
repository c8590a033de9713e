"""Build the in-tree C-ABI library ``libgqa_attn.so`` for sm_103a with nvcc.

The translation units are compiled in parallel and linked into one shared library
(CUDA runtime linked statically, no libcuda link: the driver entry point for tensor-map
encoding is looked up at run time, so the library also loads on a machine without a GPU).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libgqa_attn.so")

SOURCES = ["gqa_abi.cu", "gemm_launch.cu", "attn_launch.cu", "norm.cu", "decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libgqa_attn.so")


def _inputs_mtime() -> float:
    src = (".cu", ".cuh", ".h")
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(src)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(src)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if stale) and return the path of libgqa_attn.so."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _inputs_mtime():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([cc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        outs = list(ex.map(_run, cmds))
    if verbose:
        for o in outs:
            print(o)
    tmp = LIB_PATH + ".tmp"
    _run([cc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=("-Xptxas", "-v") if "--ptxas" in sys.argv else ()))
