"""Build libmoe_permute.so (the C-ABI CUDA library) in-tree with nvcc, and
beside it libmoe_permute_debug.so, the same sources with -DMOE_DEBUG_HOOKS
(the test hook of include/moe_permute_debug.h).  The two compile in parallel.

Usage: python -m moe_token_permute_gb300.build [--verbose]
Target: sm_103a only (GB300).  The libraries are linked against the shared
CUDA runtime so they share one runtime with the host process.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmoe_permute.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libmoe_permute_debug.so")
SOURCES = ["moe_permute_api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_permute.so")


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(root, sub)
        if glob.glob(os.path.join(d, "libcudart.so*")):
            return d
    return os.path.join(root, "lib64")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += glob.glob(os.path.join(CSRC, "*.cuh"))
    files += glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return files


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _command(nvcc: str, out: str, defines, verbose: bool):
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", *defines,
           "-I", INCLUDE, "-I", CSRC, "-cudart", "shared",
           "-Xlinker", "-rpath," + _cuda_lib_dir(nvcc),
           "-o", out] + [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the libraries that are missing or older than their sources
    (both nvcc runs in parallel); returns the production library's path."""
    targets = [(LIB_PATH, []), (DEBUG_LIB_PATH, ["-DMOE_DEBUG_HOOKS"])]
    todo = [(path, d) for path, d in targets if force or not up_to_date(path)]
    if not todo:
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    jobs = []
    for path, defines in todo:
        tmp = path + f".tmp{os.getpid()}"
        jobs.append((subprocess.Popen(_command(nvcc, tmp, defines, verbose)), tmp, path))
    failed = []
    for proc, tmp, path in jobs:
        if proc.wait() != 0:
            failed.append(path)
        else:
            os.replace(tmp, path)
    if failed:
        raise RuntimeError(f"nvcc failed building {', '.join(failed)}")
    return LIB_PATH


C_LATENCY_SOURCE = os.path.join(PKG, "c_latency.c")
C_LATENCY_PATH = os.path.join(OUT_DIR, "moe_c_latency")


def build_c_latency() -> str:
    """Compile the C latency probe (c_latency.c) against the library and the
    CUDA runtime with the host C compiler; returns the executable's path."""
    build()
    exe = C_LATENCY_PATH
    if os.path.exists(exe) and all(os.path.getmtime(f) <= os.path.getmtime(exe)
                                   for f in (C_LATENCY_SOURCE, LIB_PATH)):
        return exe
    nvcc = _nvcc()
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    cudart_dir = _cuda_lib_dir(nvcc)
    tmp = exe + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-I", cuda_inc,
         C_LATENCY_SOURCE, "-L", OUT_DIR, "-lmoe_permute", "-L", cudart_dir, "-lcudart",
         f"-Wl,-rpath,{OUT_DIR}:{cudart_dir}", "-o", tmp])
    os.replace(tmp, exe)
    return exe


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv))
