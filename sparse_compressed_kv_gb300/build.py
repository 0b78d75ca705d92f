"""Build libcsa.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel to an object
file under ``_build/``, then linked into ``sparse_compressed_kv_gb300/libcsa.so``
(static CUDA runtime, no libcuda link: the tensor-map encoder is reached
through the runtime's driver entry point).
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libcsa.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcsa.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "csa.h"))
    return hs


def _flags(verbose_ptxas: bool):
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr", "-Xcompiler", "-Wall"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    srcs = sources()
    newest = max(os.path.getmtime(p) for p in srcs + headers() + [os.path.abspath(__file__)])
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [cc] + _flags(verbose_ptxas) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    failed = [r for r in results if r[2].returncode != 0]
    for src, _, r in results:
        if r.stdout.strip() or r.stderr.strip():
            sys.stderr.write(f"--- {os.path.basename(src)}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f[0]) for f in failed))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [r[1] for r in results] + ["-cudart", "static"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
