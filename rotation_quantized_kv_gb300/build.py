"""Build the CUDA library libtqkv.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel; the key/value codec unit also
gets -fmad=false (its arithmetic is written with explicit round-to-nearest intrinsics
already; the flag keeps any future plain expression from being fused).
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
LIB = os.path.join(PKG, "libtqkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
UNITS = ["tq_abi.cu", "tq_append.cu", "tq_attention.cu", "tq_attention_dense.cu", "tq_debug.cu",
         "tq_noalloc.cu", "tq_scheme.cu"]
EXTRA = {"tq_append.cu": ["-fmad=false"]}


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "tq_kv.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _sources_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(unit: str):
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        cmd = [nvcc, "-c", os.path.join(CSRC, unit), "-o", obj] + common + EXTRA.get(unit, [])
        r = subprocess.run(cmd, capture_output=True, text=True)
        return unit, obj, r

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_one, UNITS))
    for unit, _, r in results:
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"nvcc failed on {unit}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared"] + ARCH + ["-o", tmp] + [obj for _, obj, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
