"""Compile the CUDA library in-tree: diffusion_transformer_denoiser_gb300/libmi_block.so.

Each translation unit is compiled for sm_103a in parallel, then linked into one shared library
with the C ABI of include/mi_block.h.  `python -m diffusion_transformer_denoiser_gb300._build`
rebuilds it; pass `--ptxas-v` to print register / shared-memory usage of every kernel.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmi_block.so")
SOURCES = ["api.cu", "gemm.cu", "attention.cu", "elementwise.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(ptxas_v: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "-I" + os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if ptxas_v:
        f += ["-Xptxas", "-v"]
    return f


def _stale(srcs, out) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = [os.path.join(CSRC, s) for s in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "mi_block.h")]
    return any(os.path.getmtime(d) > t for d in deps + list(srcs))


def build(force: bool = False, ptxas_v: bool = False, verbose: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not ptxas_v and not _stale(srcs, LIB):
        return LIB
    flags = _flags(ptxas_v)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    for obj, err in results:
        if (ptxas_v or verbose) and err:
            sys.stderr.write(err)
    tmp = LIB + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results] + ["-lcudart_static", "-lrt", "-lpthread", "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    out = build(force="--force" in sys.argv or "--ptxas-v" in sys.argv, ptxas_v="--ptxas-v" in sys.argv,
                verbose=True)
    print(out)
