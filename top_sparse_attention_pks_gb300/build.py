"""Builds libpks.so in-tree with nvcc for sm_103a (GB300).

``python -m top_sparse_attention_pks_gb300.build`` or ``build_library()``.
Translation units compile in parallel into ``_build/`` next to this file and
link into ``_lib/libpks.so``.  Nothing is installed outside the source tree.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIBDIR = PKG / "_lib"
LIB = LIBDIR / "libpks.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["pks_host.cpp", "k_indexer.cu", "k_topk.cu", "k_attention.cu", "k_residency.cu",
           "k_mla.cu", "k_stage.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = Path(cand) / "bin" / "nvcc"
        if cand and p.exists():
            return str(p)
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpks")
    return found


def _compile(src: Path, obj: Path, verbose: bool) -> str:
    cmd = [nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O3",
           f"-I{INCLUDE}", f"-I{CSRC}", "-c", str(src), "-o", str(obj)]
    if src.suffix == ".cu":
        cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src.name}:\n{res.stdout}\n{res.stderr}")
    return res.stderr


def _stale(obj: Path, src: Path) -> bool:
    if not obj.exists():
        return True
    deps = [src, CSRC / "pks_internal.h", INCLUDE / "pks.h"]
    return obj.stat().st_mtime < max(d.stat().st_mtime for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> Path:
    BUILD.mkdir(exist_ok=True)
    LIBDIR.mkdir(exist_ok=True)
    objs, jobs = [], []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for name in SOURCES:
            src = CSRC / name
            obj = BUILD / (name + ".o")
            objs.append(obj)
            if force or _stale(obj, src):
                jobs.append((name, ex.submit(_compile, src, obj, verbose)))
        for name, fut in jobs:
            log = fut.result()
            if verbose and log.strip():
                print(f"--- {name}\n{log}", file=sys.stderr)
    if force or jobs or not LIB.exists():
        tmp = LIB.with_suffix(f".{os.getpid()}.tmp")
        cmd = [nvcc(), "-shared", *ARCH, "-o", str(tmp), *map(str, objs)]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
