"""Build ``libpskv.so`` in-tree: every CUDA source compiled for sm_103a with nvcc,
in parallel, then linked into one shared library (static CUDA runtime).

Usage: ``python -m paged_split_kv_attn_gb300.build [--force] [--verbose-ptxas]``.
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
LIB = os.path.join(PKG, "libpskv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++20", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]
SOURCES = ["attn_tc.cu", "attn_verify.cu", "partial_mma.cu", "partial_mma_nt2.cu",
           "partial_mma_tree.cu", "partial_simt_f32.cu",
           "partial_simt_bf16.cu", "merge.cu", "append.cu", "prep.cu", "pskv_api.cu",
           "pskv_plan.cpp", "pskv_static.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpskv.so")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pskv.h"))
    files.append(os.path.abspath(__file__))
    return files


def _up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, verbose_ptxas: bool, extra: list[str], build_dir: str) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd = [nvcc(), *FLAGS, *extra, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj]
    elif verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{res.stdout}{res.stderr}")
    return obj, res.stdout + res.stderr


def build(force: bool = False, verbose_ptxas: bool = False, defines: dict | None = None,
          out: str = LIB) -> str:
    """Compile and link the library unless it is newer than every source; return its path.

    ``defines`` sets the compile-time tuning macros (for example
    ``{"PSKV_MMA_STAGES": 4}``); a build with defines goes to ``out`` and is
    always rebuilt."""
    extra = [f"-D{k}={v}" for k, v in (defines or {}).items()]
    if not force and not verbose_ptxas and not extra and out == LIB and _up_to_date():
        return LIB
    build_dir = BUILD if out == LIB else out + ".objs"
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, extra, build_dir), SOURCES))
    if verbose_ptxas:
        for _, log in results:
            sys.stdout.write(log)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{res.stdout}{res.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv))
