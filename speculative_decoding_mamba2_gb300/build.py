"""Build libssmtree.so (sm_103a) in-tree with nvcc.

    python -m speculative_decoding_mamba2_gb300.build

Objects and the library go to ``_build/<machine>/`` inside this package, so an
x86 build and an aarch64 build never mix.  Translation units compile in
parallel; an up-to-date library is not rebuilt.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
SOURCES = ["api.cu", "verify.cu", "verify_tc.cu", "commit.cu", "draft.cu", "noalloc.cu", "chain.cu", "gemm.cu", "norm.cu",
           "layer_api.cu", "draft_tree.cu", "selftest.cu", "layout.cpp"]
HEADERS = [os.path.join(CSRC, h) for h in ("common.cuh", "draft_tree.cuh", "log_apply.cuh", "tc.cuh")] + \
    [os.path.join(INCLUDE, h) for h in ("ssm_tree.h", "ssm_layer.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
LIBNAME = "libssmtree.so"


def build_dir() -> str:
    return os.path.join(PKG, "_build", platform.machine())


def lib_path() -> str:
    return os.path.join(build_dir(), LIBNAME)


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put /usr/local/cuda/bin on PATH)")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout.strip() or r.stderr.strip()):
        print(r.stdout, r.stderr, sep="\n", flush=True)
    return r


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every translation unit for sm_103a and link libssmtree.so; returns its path."""
    nvcc = _nvcc()
    out = build_dir()
    os.makedirs(out, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE, "-I", CSRC]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out, os.path.splitext(src)[0] + ".o")
        if force or ptxas_verbose or _stale(o, [s] + HEADERS):
            lang = ["-x", "cu"] if src.endswith(".cu") else ["-x", "c++"]
            jobs.append([nvcc] + flags + lang + ["-c", s, "-o", o])
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            results = list(ex.map(lambda c: _run(c, verbose), jobs))
        if ptxas_verbose:
            for r in results:
                print(r.stderr)
    objs = [os.path.join(out, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    lib = lib_path()
    if force or jobs or _stale(lib, objs):
        _run([nvcc] + ARCH + ["-shared", "-o", lib] + objs + ["-cudart", "static"], verbose)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas-v" in sys.argv))
