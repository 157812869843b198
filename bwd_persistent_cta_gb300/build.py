"""Build librnn.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel into ``_build/`` next to this file;
the shared library lands beside this file as ``librnn.so``.  No cmake, no
torch extension machinery: plain nvcc, so the same command works on the x86
build host (cross-compiling device code) and on the Arm GPU hosts.
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
LIB = os.path.join(HERE, "librnn.so")
SOURCES = ["api.cpp", "tmap.cpp", "layout.cu", "gemm_simt.cu", "gemm_tc.cu",
           "persist_simt.cu", "persist_tc.cu", "persist_tc_fwd.cu", "persist_tc_bwd.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool = False, extra=()):
    f = list(extra) + ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
                "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _compile(src: str, verbose_ptxas: bool, build_dir: str = BUILD, extra=()) -> str:
    obj = os.path.join(build_dir, src + ".o")
    cmd = [nvcc()] + _flags(verbose_ptxas, extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd = [nvcc(), "-x", "cu"] + cmd[1:]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, extra_flags=(), lib_path: str = LIB,
          build_dir: str = BUILD) -> str:
    """Compile (if any source is newer than the library) and return its path.
    ``extra_flags`` / ``lib_path`` / ``build_dir`` build a variant elsewhere
    (e.g. with -D switches for latency studies) without touching the default."""
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(ROOT, "include", h) for h in os.listdir(os.path.join(ROOT, "include"))]
    if not force and os.path.exists(lib_path):
        lib_t = os.path.getmtime(lib_path)
        if all(os.path.getmtime(d) <= lib_t for d in deps):
            return lib_path
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, build_dir, extra_flags), SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
