"""Builds libfa.so (the C-ABI attention library) in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled on its own (in parallel), then linked
into ``exact_attention_05_gb300/_build/libfa.so`` with the CUDA runtime linked
statically and every symbol except the ``fa_*`` C ABI hidden.  No GPU is
needed: nvcc cross-compiles.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD, "libfa.so")
SOURCES = ["fa_api.cu", "fa_prefill.cu", "fa_backward.cu", "fa_decode.cu", "fa_decode_fp8.cu", "fa_decode_paged.cu",
           "fa_decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers():
    out = [os.path.join(INCLUDE, "fa.h")]
    out += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return out


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if not _stale(obj, [path] + _headers()):
        return obj
    cmd = [_nvcc(), "-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler",
           "-fPIC,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC, "-c", path, "-o", obj + ".tmp"]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas:
        sys.stderr.write(res.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool | None = None) -> str:
    """Compile and link libfa.so if any source is newer than it; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    if verbose_ptxas is None:
        verbose_ptxas = os.environ.get("FA_PTXAS_VERBOSE", "") == "1"
    if force:
        for f in os.listdir(BUILD):
            if f.endswith((".o", ".so")):
                os.remove(os.path.join(BUILD, f))
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    if _stale(LIB_PATH, objs):
        cmd = [_nvcc(), "-shared", *ARCH, *objs, "-o", LIB_PATH + ".tmp", "-Xlinker",
               "--exclude-libs,ALL", "-Xlinker", "-Bsymbolic"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(LIB_PATH + ".tmp", LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
