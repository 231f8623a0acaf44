"""Compiles the C-ABI library libzero_gb300.so (CUDA kernels + host API) for sm_103a.

Two translation units are compiled in parallel with nvcc and linked into
zero_gradient_reduce_scatter_gb300/_build/libzero_gb300.so (in-tree, git-ignored). The CUDA
runtime is linked as a shared library so that a process that also uses PyTorch runs a
single runtime instance (same soname).
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libzero_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
# The bounds-checked variant (every kernel index tested before use; for tests).
CHECKED_LIB_PATH = os.path.join(BUILD_DIR, "libzero_gb300_checked.so")

SOURCES = ["zero_kernels.cu", "zero_api.cpp", "zero_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero_gb300.so")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, "zero_internal.h"), os.path.join(INCLUDE, "zero_gb300.h"), __file__]
    return files


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Build libzero_gb300.so (or, with checked=True, the bounds-checked
    libzero_gb300_checked.so) if missing or older than its sources; returns its path."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and not is_stale(lib_path):
        return lib_path
    nvcc = _nvcc()
    obj_dir = os.path.join(BUILD_DIR, "checked" if checked else "release")
    os.makedirs(obj_dir, exist_ok=True)
    common = ["-std=c++17", "-O3", "-lineinfo", "-I", INCLUDE, "-I", CSRC,
              "-Xcompiler", "-fPIC,-ffp-contract=off,-fno-fast-math,-Wall"]
    if checked:
        common.append("-DZERO_CHECKED")
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = [nvcc, *common, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{out}")
        if verbose and out.strip():
            print(out)
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", f"-rpath,{_cuda_lib_dir(nvcc)}"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}")
    os.replace(tmp, lib_path)
    return lib_path
