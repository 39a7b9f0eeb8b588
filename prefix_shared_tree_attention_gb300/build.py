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
# TPA_DEBUG build: kernels check every metadata index they read from a tree
# view before using it as an address and report a bad one through the status
# word (TPA_ERR_INVALID_ARG) instead of touching memory with it
DEBUG_OBJ_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libtpa_debug.so")

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


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(p) > t for p in _deps())


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")


def _jobs(obj_dir: str, extra_nvcc: list[str]) -> list[tuple[str, list[str]]]:
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        jobs.append((obj, [nvcc, *ARCH, "-lineinfo", *common, "-Xcompiler", "-fPIC", *extra_nvcc, "-c",
                           os.path.join(CSRC, src), "-o", obj]))
    cxx = shutil.which("g++") or "g++"
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")  # NVTX headers
    for src in HOST_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        jobs.append((obj, [cxx, *common, "-isystem", cuda_inc, "-fPIC", "-Wall", "-c", os.path.join(CSRC, src),
                           "-o", obj]))
    return jobs


def build(force: bool = False, verbose: bool = False, extra_nvcc: list[str] | None = None,
          debug: bool = False) -> str:
    """Compile and link libtpa.so if any source is newer than it; returns its
    path.  With ``debug`` also libtpa_debug.so (TPA_DEBUG=1); both variants
    compile in one pool of jobs."""
    variants = [(OBJ_DIR, LIB_PATH, list(extra_nvcc or []))]
    if debug:
        variants.append((DEBUG_OBJ_DIR, DEBUG_LIB_PATH, list(extra_nvcc or []) + ["-DTPA_DEBUG=1"]))
    todo = [v for v in variants if force or is_stale(v[1])]
    if not todo:
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    jobs = []
    for obj_dir, _, flags in todo:
        os.makedirs(obj_dir, exist_ok=True)
        jobs += _jobs(obj_dir, flags)
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        list(ex.map(lambda j: _run(j[1]), jobs))
    nvcc = _nvcc()
    for obj_dir, path, _ in todo:
        objs = [os.path.join(obj_dir, s + ".o") for s in CUDA_SOURCES + HOST_SOURCES]
        tmp = path + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, path)
        if verbose:
            print(f"built {path}", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
