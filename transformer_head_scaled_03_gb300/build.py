"""Build libmha_gb300.so in-tree with nvcc for sm_103a (no cmake).

Each .cu file compiles to an object in parallel, then nvcc links the shared
library (CUDA runtime linked statically; the TMA descriptor encoder is found
through the runtime's driver entry point, so no -lcuda).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmha_gb300.so")
SOURCES = ["mha_api.cu", "sdpa_bf16.cu", "gemm_bf16.cu", "gemm_ln_bf16.cu", "fp32_path.cu",
           "mha_noalloc.cu",
           "layernorm.cu", "encoder_api.cu", "sdpa_decode.cu",
           "embed_pe.cu", "sdpa_backward.cu", "host_pipeline.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
                "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _inputs_mtime() -> float:
    paths = [os.path.join(CSRC, s) for s in os.listdir(CSRC)]
    paths += [os.path.join(INCLUDE, s) for s in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _inputs_mtime()


def build(force: bool = False, verbose: bool = False, log=None) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = _flags(verbose)

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if log is not None:
        for (_, err), src in zip(results, SOURCES):
            if err.strip():
                log.write(f"== {src}\n{err}\n")
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, log=sys.stderr))
