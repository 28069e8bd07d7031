"""Build librmsnorm_gb300.so in-tree with nvcc for sm_103a.

The translation units compile in parallel (one nvcc per file) into
``_build/`` and link into ``librmsnorm_gb300.so`` next to this file. The
CUDA runtime is linked statically so the library loads without a matching
libcudart on the library path; it shares the device's primary context with
any other CUDA user in the process (device pointers and streams from
PyTorch are valid in it).

Usage:  python -m row_wise_normalization_rmsnorm_gb300.build [--force]
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
LIB = os.path.join(HERE, "librmsnorm_gb300.so")
HEADER = os.path.join(ROOT, "include", "rmsnorm.h")

SOURCES = ["api.cu", "fwd_bf16.cu", "fwd_f32.cu", "fwd_f16.cu", "fwd_bf16w32.cu", "fwd_f16w32.cu",
           "fwd8_bf16.cu", "fwd8_f16.cu", "fwd8_f32.cu", "fwd8_bf16w32.cu", "fwd8_f16w32.cu", "ln_bf16.cu", "ln_f16.cu", "ln_f32.cu", "ln_bf16w32.cu", "ln_f16w32.cu",
           "bwd_bf16.cu", "bwd_f32.cu", "bwd_f16.cu", "bwd_bf16w32.cu", "bwd_f16w32.cu",
           "fwd_peel_f32.cu", "fwd_peel_bf16.cu", "fwd_peel_f16.cu", "bwd_peel_f32.cu", "bwd_peel_bf16.cu",
           "bwd_peel_f16.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "plans.h", "fwd_kernels.cuh", "bwd_kernels.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librmsnorm_gb300.so")


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else 0.0


def _stale(force: bool) -> bool:
    if force or not os.path.exists(LIB):
        return True
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [HEADER, os.path.abspath(__file__)]
    return max(_mtime(p) for p in deps) > _mtime(LIB)


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile (if any source changed) and return the library path."""
    if not _stale(force):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra or [])
    if verbose:
        extra += ["-Xptxas", "-v"]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "--cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
