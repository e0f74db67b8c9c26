"""Builds libpagedkv.so in-tree for sm_103a with nvcc.

Each source compiles to its own object in parallel (one -gencode, so a build
takes well under a minute), then nvcc links them into the shared library next
to this file. The library links the CUDA runtime dynamically, so it shares the
runtime that PyTorch loads.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libpagedkv.so")
SOURCES = ["attention.cu", "cache_ops.cu", "block_manager.cpp", "decode_step.cpp", "allocator_sim.cpp"]
HEADERS = [os.path.join(CSRC, "pk_device.cuh"), os.path.join(INCLUDE, "pagedkv.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

_lock = threading.Lock()


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    for cand in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libpagedkv")


def _cuda_lib_dir(nvcc: str) -> Optional[str]:
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib"):
        d = os.path.join(home, sub)
        if os.path.isdir(d):
            return d
    return None


def _stale(target: str, deps: List[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def compile_flags(ptxas_verbose: bool = False) -> List[str]:
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
             "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    return flags


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile (if stale) and link libpagedkv.so; returns its path."""
    with _lock:
        nvcc = nvcc_path()
        os.makedirs(BUILD_DIR, exist_ok=True)
        srcs = [os.path.join(CSRC, s) for s in SOURCES]
        objs = [os.path.join(BUILD_DIR, s + ".o") for s in SOURCES]
        todo = [(s, o) for s, o in zip(srcs, objs) if force or ptxas_verbose or _stale(o, [s] + HEADERS)]

        def compile_one(so):
            src, obj = so
            cmd = [nvcc, *compile_flags(ptxas_verbose), "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
            return r.stdout + r.stderr

        if todo:
            with ThreadPoolExecutor(max_workers=len(todo)) as ex:
                logs = list(ex.map(compile_one, todo))
            if verbose or ptxas_verbose:
                for log in logs:
                    if log.strip():
                        print(log)
        if todo or force or _stale(LIB_PATH, objs):
            libdir = _cuda_lib_dir(nvcc)
            tmp = LIB_PATH + f".tmp{os.getpid()}"
            cmd = [nvcc, ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
            if libdir:
                cmd += ["-Xlinker", f"-rpath={libdir}"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, LIB_PATH)
        return LIB_PATH


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
