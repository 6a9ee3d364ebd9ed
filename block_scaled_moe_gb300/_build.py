"""Build of libblockmoe.so: nvcc for sm_103a, translation units compiled in parallel.

Variant "bounds" builds libblockmoe_bounds.so with -DMOE_DEBUG_BOUNDS: every index the kernels compute
into the workspace or an output row is checked, a miss is recorded in the status word and skipped.
Variant "trace" builds libblockmoe_trace.so with -DBMOE_TRACE: the kernels stamp clocks into trace
buffers that block_scaled_moe_gb300.trace reads back.  The binding loads a variant when
BMOE_LIB_VARIANT names it."""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
VARIANTS = {"": [], "bounds": ["-DMOE_DEBUG_BOUNDS"], "trace": ["-DBMOE_TRACE"]}
SOURCES = ["moe_api.cu", "moe_kernels.cu", "moe_gemm.cu", "moe_fused.cu", "moe_noalloc.cu", "moe_route.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-Wall", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr", "-Werror", "all-warnings"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libblockmoe.so")
    return cand


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "blockmoe.h")]
    return max(os.path.getmtime(f) for f in files)


def lib_path(variant: str = "") -> str:
    return os.path.join(PKG, "lib", f"libblockmoe_{variant}.so" if variant else "libblockmoe.so")


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    if variant not in VARIANTS:
        raise ValueError(f"unknown build variant {variant!r}; known: {sorted(VARIANTS)}")
    LIB = lib_path(variant)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps() and not extra_flags:
        return LIB
    bdir = os.path.join(BUILD, variant) if variant else BUILD
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *FLAGS, *VARIANTS[variant], *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
