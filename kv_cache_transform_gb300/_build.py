"""Build libkvtc.so in-tree with nvcc for sm_103a (no CMake, no torch)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libkvtc.so")
BUILD = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
         "-I" + os.path.join(ROOT, "include")]
SOURCES = ["kvtc_host.cu", "kvtc_kernels.cu", "kvtc_calib.cu",
           "kvtc_static.cu", "kvtc_fieldpack.cu"]
LIBS = ["-lcusolver"]
DEPS = SOURCES + ["kvtc_internal.cuh", "ptx.cuh"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date() -> bool:
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    srcs = [os.path.join(CSRC, f) for f in DEPS]
    srcs.append(os.path.join(ROOT, "include", "kvtc.h"))
    return all(os.path.getmtime(s) <= t for s in srcs)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel and link the library."""
    if not force and up_to_date():
        return OUT
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = OUT + ".tmp"
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs, *LIBS]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force=True, verbose=True))
