"""Build libcpring.so in-tree with nvcc for sm_103a.

Sources are compiled in parallel (one nvcc process per translation unit)
and linked into context_ring_attention_fwd_gb300/_lib/libcpring.so.  Object
files go to context_ring_attention_fwd_gb300/_lib/obj/.  Nothing here needs a
GPU: nvcc cross-compiles.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libcpring.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

SOURCES = ["attn_sm103.cu", "attn_f32.cu", "merge.cu", "noalloc.cu", "ring_emulation.cpp",
           "ulysses.cu", "fp8.cu", "attn_bwd_sm103.cu", "api.cpp", "scratch.cpp",
           "host_path.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcpring.so")


# The tensor-core kernel moves registers between its warpgroups with
# setmaxnreg; the split is sized for exactly this many registers per thread at
# launch, so a build that comes out different is refused (the split would not
# fit and the kernel would stall).
SPLIT_KERNELS = ("ring_attn_bf16_kernel", "ring_attn_fp8_kernel", "ring_attn_bwd_kernel")
SPLIT_LAUNCH_REGS = 168


def _check_split(src: str, ptxas_log: str) -> None:
    entry = None
    for line in ptxas_log.splitlines():
        if "Compiling entry function" in line:
            entry = line
        elif "Used" in line and "registers" in line and entry and \
                any(k in entry for k in SPLIT_KERNELS):
            n = int(line.split("Used")[1].split("registers")[0])
            if n != SPLIT_LAUNCH_REGS:
                raise RuntimeError(f"{src}: {entry.strip()} launches with {n} registers per "
                                   f"thread, its register split needs {SPLIT_LAUNCH_REGS}")
            entry = None


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OBJDIR, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cu"):
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if src.endswith(".cu"):
        _check_split(src, r.stdout + r.stderr)
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(verbose: bool = False) -> str:
    """Compile every source and link libcpring.so; returns its path."""
    os.makedirs(OBJDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
