"""Build libtpa.so in-tree: every translation unit compiled in parallel with
nvcc for sm_103a (the host packer with g++), then linked into one shared
library next to this file (``_lib/libtpa.so``)."""
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
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtpa.so")

CUDA_SOURCES = ["runtime.cu", "classify.cu", "logprobs.cu", "attn_fwd.cu", "attn_bwd.cu", "dense_mask.cu", "lm_head.cu"]
HOST_SOURCES = ["pack.cpp", "balance.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtpa")
    return cand


def _deps() -> list[str]:
    out = [os.path.join(INCLUDE, "tpa.h")]
    for f in os.listdir(CSRC):
        out.append(os.path.join(CSRC, f))
    return out


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _deps())


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")


def build(force: bool = False, verbose: bool = False, extra_nvcc: list[str] | None = None) -> str:
    """Compile and link libtpa.so if any source is newer than it; returns its path."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(OBJ_DIR, src + ".o")
        jobs.append((obj, [nvcc, *ARCH, "-lineinfo", *common, "-Xcompiler", "-fPIC",
                           *(extra_nvcc or []), "-c", os.path.join(CSRC, src), "-o", obj]))
    cxx = shutil.which("g++") or "g++"
    for src in HOST_SOURCES:
        obj = os.path.join(OBJ_DIR, src + ".o")
        jobs.append((obj, [cxx, *common, "-fPIC", "-Wall", "-c", os.path.join(CSRC, src), "-o", obj]))
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        list(ex.map(lambda j: _run(j[1]), jobs))
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[j[0] for j in jobs]])
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(f"built {LIB_PATH}", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
