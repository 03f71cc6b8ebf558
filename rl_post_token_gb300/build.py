"""Build ``libgrpo.so`` in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own process (in parallel), then nvcc links the shared
library with the static CUDA runtime, so the library loads on a machine without a GPU and
needs no libcudart at run time. Objects go to ``rl_post_token_gb300/_build/``, with each CUDA
file's ptxas resource report (registers, spills per kernel) beside its object as
``<source>.ptxas.txt``.

    python -m rl_post_token_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgrpo.so")

SOURCES = ["grpo_plan.cpp", "grpo_window.cpp", "grpo_rowpass.cu", "grpo_step.cu", "grpo_lmhead.cu"]
LINK: list = []  # every kernel is the library's own: no CUDA library beyond the static runtime
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgrpo.so")


def _deps():
    files = [os.path.join(CSRC, s) for s in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, h) for h in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def ptxas_report(src: str) -> str:
    """Path of the ptxas resource report of a CUDA source from the last build."""
    return os.path.join(BUILD, src + ".ptxas.txt")


def _up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    if not all(os.path.exists(ptxas_report(s)) for s in SOURCES if s.endswith(".cu")):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, verbose: bool) -> str:
    nvcc = _nvcc()
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    common = ["-O3", "-std=c++17", f"-I{INCLUDE}", f"-I{CSRC}", "-Xcompiler", "-fPIC,-fvisibility=hidden"]
    if src.endswith(".cu"):
        cmd = [nvcc, *ARCH, "-Xptxas=-v", "-lineinfo", "--expt-relaxed-constexpr", *common, "-c", path, "-o", obj]
    else:
        cmd = [nvcc, "-x", "c++", *common, "-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compiling {src} failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if src.endswith(".cu"):
        with open(ptxas_report(src), "w") as f:
            f.write(r.stdout + r.stderr)
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if any source changed; return its path."""
    if not force and _up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, *LINK]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
