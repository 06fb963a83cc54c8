"""Build libkvx.so (the C-ABI library) in-tree for sm_103a with nvcc.

Three translation units, compiled in parallel: the CUDA kernels + entry points (kvx.cu, by
nvcc), the host logic (kvx_host.cpp) and the SM partitioning (kvx_partition.cpp), the last
two by the host C++ compiler.  The CUDA runtime is
linked statically so the library loads on machines without a GPU (its host logic and
exported symbols stay usable there).
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
LIB = os.path.join(PKG, "libkvx.so")
BUILD_DIR = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = [os.path.join(CSRC, f) for f in ("kvx.cu", "kvx_kernels.cuh", "kvx_host.cpp",
                                             "kvx_partition.cpp", "kvx_internal.h")]
HEADER = os.path.join(ROOT, "include", "kvx.h")


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in SOURCES + [HEADER])


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libkvx.so if a source is newer than it (or force); return its path."""
    if not force and not _stale():
        return LIB
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    inc = os.path.join(home, "include")
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f"{os.getpid()}"
    obj_cu = os.path.join(BUILD_DIR, f"kvx.{tag}.o")
    cu = [nvcc, "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xptxas", "-v", "-Xcompiler", "-fPIC",
          "-c", os.path.join(CSRC, "kvx.cu"), "-o", obj_cu]
    cxx = shutil.which("g++") or shutil.which("c++")
    objs = [obj_cu]
    cmds = [cu]
    for src in ("kvx_host.cpp", "kvx_partition.cpp"):
        obj = os.path.join(BUILD_DIR, f"{src[:-4]}.{tag}.o")
        objs.append(obj)
        cmds.append([cxx, "-O2", "-std=c++17", "-fPIC", f"-I{inc}", "-c",
                     os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(len(cmds)) as ex:
        logs = list(ex.map(_run, cmds))
    tmp = LIB + f".tmp{tag}"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    for o in objs:
        os.remove(o)
    if verbose:
        sys.stdout.write(logs[0])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
