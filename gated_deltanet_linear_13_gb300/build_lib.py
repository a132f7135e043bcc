"""Build libgdn.so in-tree: every csrc/*.cu for sm_103a, compiled in parallel, then linked.

    python -m gated_deltanet_linear_13_gb300.build_lib [--force] [--bounds-check]

--bounds-check builds libgdn_checked.so instead: the same library compiled with
-DGDN_BOUNDS_CHECK, whose kernels check their computed global indices and record
GDN_ERR_DEVICE_INDEX (skipping the access) instead of faulting.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgdn.so")
LIB_CHECKED = os.path.join(PKG, "libgdn_checked.so")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", INCLUDE, "-I", CSRC]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "gdn.h")]


def _up_to_date(lib: str) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, extra, bdir: str) -> str:
    obj = os.path.join(bdir, os.path.basename(src) + ".o")
    cmd = [NVCC] + ARCH + FLAGS + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, extra_flags=(), checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    bdir = os.path.join(BUILD, "checked") if checked else BUILD
    flags = list(extra_flags) + (["-DGDN_BOUNDS_CHECK"] if checked else [])
    if not force and not extra_flags and _up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, bdir), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, checked="--bounds-check" in sys.argv))
