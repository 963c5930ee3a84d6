"""Build libmhc.so (the seam's C-ABI library) in-tree with nvcc for sm_103a.

Each CUDA translation unit under ``csrc/`` is compiled in parallel to an
object file, then linked into ``_build/libmhc.so`` (CUDA runtime linked
statically, so loading the library needs no GPU).  Rebuilds only what
changed.  Usage: ``python -m mhc_hyper_connection_pre_gb300.build [--ptxas-v]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmhc.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmhc.so")


def _newest_dep_mtime() -> float:
    deps = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(d) for d in deps), default=0.0)


def _compile(src: str, ptxas_v: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    dep_t = max(os.path.getmtime(src), _newest_dep_mtime())
    if not ptxas_v and os.path.exists(obj) and os.path.getmtime(obj) >= dep_t:
        return obj, ""
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj + ".tmp"]
    if ptxas_v:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj, r.stderr


def build(ptxas_v: bool = False, force: bool = False) -> str:
    """Compile every ``csrc/*.cu`` and link ``_build/libmhc.so``; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for o in glob.glob(os.path.join(BUILD, "*.o")):
            os.remove(o)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_v), srcs))
    if ptxas_v:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    newest = max(os.path.getmtime(o) for o in objs)
    if force or ptxas_v or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libmhc.so failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(ptxas_v="--ptxas-v" in sys.argv, force="--force" in sys.argv))
