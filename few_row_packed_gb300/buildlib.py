"""Builds the in-tree CUDA library liblbv.so for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into
few_row_packed_gb300/liblbv.so (git-ignored).  No cmake, no torch extension
machinery: the library is a plain C ABI (include/lbv.h).

build(checked=True) makes liblbv_checked.so instead: the same sources with
LBV_CHECKED defined, whose kernels check their copy and buffer ranges, record
a bounds error in the plan's status word and skip the access (the release
library's device code is unchanged by those checks).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "liblbv.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "liblbv_checked.so")

SOURCES = [
    "api.cpp",
    "tc_api.cpp",
    "t8_api.cpp",
    "aux_kernels.cu",
    "verify_sign1.cu",
    "verify_affine2_g32.cu",
    "verify_affine2_g64.cu",
    "verify_affine2_g128.cu",
    "verify_q4_0.cu",
    "fused_aux.cu",
    "tc_aux.cu",
    "tc_sign1.cu",
    "tc_affine2_g32.cu",
    "tc_affine2_g64.cu",
    "tc_affine2_g128.cu",
    "tc_q4_0.cu",
    "t8_sign1.cu",
    "t8_affine2_g128.cu",
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "-Xcompiler", "-fvisibility=hidden",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblbv.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "lbv.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib, bdir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = FLAGS + (["-DLBV_CHECKED"] if checked else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    jobs = min(len(SOURCES), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(jobs) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
