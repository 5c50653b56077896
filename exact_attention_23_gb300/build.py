"""Build libfa.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked with the CUDA runtime
statically, so the library's only runtime dependency is the driver (libcuda), which
the runtime opens on first use.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libfa.so")

SOURCES = ["fa_api.cu", "fa_fwd1.cu", "fa_fwd1_gen.cu", "fa_fwd_pair.cu", "fa_fwd_d64.cu", "fa_fwd_d128.cu", "fa_fwd_fp8.cu", "fa_fwd_gen_d64.cu",
           "fa_fwd_gen_d128.cu", "fa_fwd_ext_api.cu", "fa_decode.cu", "fa_bwd_d64.cu", "fa_bwd_d128.cu",
           "fa_bwd_api.cu",
           "fa_noalloc.cu", "fa_hostio.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False) -> str:
    """Compile every CUDA source and link libfa.so; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    log = "".join(err for _, err in results)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-Xlinker",
           "--version-script=" + os.path.join(CSRC, "exports.map"), "-o", tmp,
           *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        sys.stderr.write(log)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
