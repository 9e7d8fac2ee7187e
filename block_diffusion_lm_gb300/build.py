"""Build libcsbp.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel into _build/, then the
objects link into block_diffusion_lm_gb300/libcsbp.so (the CUDA runtime is
linked statically, so the library needs only the driver at run time).
Rebuilds only what changed (source or header newer than the object).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcsbp.so")
# debug variant: kernels validate their work-list records before any access
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libcsbp_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["schedule.cpp", "csbp_api.cu", "attn_fwd.cu", "attn_bwd.cu", "elementwise.cu",
           "noalloc.cu", "vocab_ce.cu", "selftest.cu"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcsbp")


def _headers_mtime() -> float:
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, src.rsplit(".", 1)[0] + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(path), _headers_mtime()):
        return obj
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-c", path, "-o", obj]
    if debug:
        cmd.insert(1, "-DCSBP_DEBUG_CHECKS")
    if src.endswith(".cu"):
        cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
    else:
        cmd += ["-x", "c++"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, debug: bool = False) -> str:
    """Compile and link libcsbp.so (or, with debug=True, libcsbp_debug.so,
    whose kernels check their work-list records); returns its path."""
    out, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(out, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), SOURCES))
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
