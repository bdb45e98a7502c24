"""Builds libssm_b300.so in-tree with nvcc for sm_103a (run: python -m selective_state_space_139_b300.build).

The library is a plain shared object with a C ABI (include/ssm.h); nothing here links PyTorch.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libssm_b300.so")
# The checked debug build: every kernel's global accesses go through index checks that report
# SSM_ERR_CHECK through ssm_device_status() instead of touching memory outside their buffers.
LIB_CHECK = os.path.join(LIB_DIR, "libssm_b300_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(INCLUDE, "ssm.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compiles each kernel file to an object in parallel, then links the shared library."""
    lib = LIB_CHECK if checked else LIB
    if not force and up_to_date(lib):
        return lib
    os.makedirs(LIB_DIR, exist_ok=True)
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-Xcompiler", "-Wall",
             "-I", INCLUDE, "-I", CSRC]
    if checked:
        flags.append("-DSSM_CHECK=1")
    if verbose:
        flags.append("-Xptxas=-v")
    with tempfile.TemporaryDirectory(prefix="ssm_obj_") as obj_dir:
        def compile_one(src: str) -> str:
            obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
            cmd = [nvcc(), *flags, "-c", "-o", obj, src]
            if verbose:
                print(" ".join(cmd))
            subprocess.check_call(cmd)
            return obj

        srcs = sources()
        with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as pool:
            objs = list(pool.map(compile_one, srcs))
        tmp = lib + ".tmp"
        subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    for chk in (False, True):
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked=chk))
