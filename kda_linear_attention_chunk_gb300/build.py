"""Ahead-of-time build of libkda.so (sm_103a) with nvcc.

Every translation unit under csrc/ is compiled in parallel to an object file
with ``-gencode arch=compute_103a,code=sm_103a``, then linked into one shared
library with the CUDA runtime linked statically.  Nothing is compiled at
import time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from typing import List, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkda.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libkda.so")


def sources() -> List[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, out_dir: str = BUILD, defines: Sequence[str] = ()) -> tuple:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, res.returncode, res.stdout + res.stderr


def _build(out_dir: str, lib: str, defines: Sequence[str], log_path: Optional[str]) -> str:
    os.makedirs(out_dir, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda src: _compile(src, out_dir, defines), srcs))
    logs, objs = [], []
    for src, obj, rc, out in results:
        logs.append(f"== {os.path.basename(src)}\n{out}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{out}")
        objs.append(obj)
    tmp = lib + ".tmp"
    res = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}{res.stderr}")
    os.replace(tmp, lib)
    with open(log_path or os.path.join(out_dir, "ptxas.log"), "w") as fh:
        fh.write("\n".join(logs))
    return lib


def build(verbose: bool = False, log_path: Optional[str] = None) -> str:
    """Compile and link libkda.so; returns its path.  Raises on failure."""
    lib = _build(BUILD, LIB, (), log_path)
    if verbose:
        print(open(log_path or os.path.join(BUILD, "ptxas.log")).read())
    return lib


def build_variant(tag: str, defines: Sequence[str]) -> str:
    """A separate copy of the library compiled with extra -D definitions, in
    _build/<tag>/ (for tests that need a kernel built differently, such as a
    wait limit of zero); returns the path of its libkda.so."""
    out_dir = os.path.join(BUILD, tag)
    return _build(out_dir, os.path.join(out_dir, "libkda.so"), tuple(defines), None)


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
           [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(p) > t for p in deps)


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
