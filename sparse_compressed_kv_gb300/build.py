"""Build libcsa.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel to an object
file under ``_build/``, then linked into ``sparse_compressed_kv_gb300/libcsa.so``
(static CUDA runtime, no libcuda link: the tensor-map encoder is reached
through the runtime's driver entry point).

``checks=True`` builds the same sources with ``CSA_CHECKS`` defined into
``libcsa_checks.so`` (objects under ``_build/checks``): internal bounds
checks that report ``CSA_DEV_CHECK`` in the status word instead of touching
memory out of range.  ``build_all()`` builds both at once.
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
LIB_CHECKS = os.path.join(HERE, "libcsa_checks.so")
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


def _variant(checks: bool):
    return (LIB_CHECKS, os.path.join(BUILD, "checks"), ["-DCSA_CHECKS=1"]) if checks else (LIB, BUILD, [])


def _stale(lib: str) -> bool:
    newest = max(os.path.getmtime(p) for p in sources() + headers() + [os.path.abspath(__file__)])
    return not os.path.exists(lib) or os.path.getmtime(lib) < newest


def _build_variants(variants, verbose_ptxas: bool, jobs):
    cc = nvcc()
    srcs = sources()
    work = []
    for checks in variants:
        lib, bdir, extra = _variant(checks)
        os.makedirs(bdir, exist_ok=True)
        for src in srcs:
            work.append((checks, src, os.path.join(bdir, os.path.basename(src) + ".o"), extra))

    def compile_one(w):
        checks, src, obj, extra = w
        cmd = [cc] + _flags(verbose_ptxas) + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return checks, src, obj, r

    with cf.ThreadPoolExecutor(max_workers=jobs or min(16, len(work))) as ex:
        results = list(ex.map(compile_one, work))
    for _, src, _, r in results:
        if r.stdout.strip() or r.stderr.strip():
            sys.stderr.write(f"--- {os.path.basename(src)}\n{r.stdout}{r.stderr}")
    failed = [r for r in results if r[3].returncode != 0]
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f[1]) for f in failed))
    for checks in variants:
        lib = _variant(checks)[0]
        objs = [r[2] for r in results if r[0] == checks]
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"], check=True)
        os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None,
          checks: bool = False) -> str:
    lib = _variant(checks)[0]
    if force or _stale(lib):
        _build_variants([checks], verbose_ptxas, jobs)
    return lib


def build_all(force: bool = False, jobs: int | None = None) -> None:
    """libcsa.so and libcsa_checks.so, compiled together."""
    variants = [c for c in (False, True) if force or _stale(_variant(c)[0])]
    if variants:
        _build_variants(variants, False, jobs)


if __name__ == "__main__":
    if "--all" in sys.argv:
        build_all(force="--force" in sys.argv)
        print(LIB, LIB_CHECKS)
    else:
        print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                    checks="--checks" in sys.argv))
