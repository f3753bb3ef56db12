"""Builds the CUDA library (libmoe_gb300) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library exporting the C ABI of include/moe_layer.h.  The output name carries
the host architecture so a build made on one machine is never loaded on
another.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
SOURCES = ["moe_abi.cu", "route_prologue.cu", "router.cu", "combine.cu", "gemm_fwd.cu", "gemm_dgrad.cu", "fp8.cu",
           "gemm_wgrad.cu", "selftest.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", "-Xptxas", "-warn-spills"]


def lib_path() -> str:
    return os.path.join(BUILD, f"libmoe_gb300_{platform.machine()}.so")


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "moe_layer.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    out = lib_path()
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    out = lib_path()
    if not force and up_to_date():
        return out
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, f"obj_{platform.machine()}")
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc] + CFLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
