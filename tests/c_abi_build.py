"""Compile the plain C consumer of the library (tests/c_abi/moe_c_consumer.c)
together with the oracle's C source, against libmoe_permute.so and the CUDA
runtime."""
from __future__ import annotations

import os
import subprocess

from moe_token_permute_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "tests", "c_abi", "moe_c_consumer.c")
ORACLE_C = os.path.join(ROOT, "oracle", "moe_oracle.c")


def cuda_root() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(cuda_build._nvcc())))


def build_consumer(out_dir: str) -> str:
    cuda_build.build()
    lib_dir = os.path.dirname(cuda_build.LIB_PATH)
    cudart_dir = cuda_build._cuda_lib_dir(cuda_build._nvcc())
    exe = os.path.join(out_dir, "moe_c_consumer")
    subprocess.check_call(
        ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-Wall", "-Wextra", "-Werror",
         "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda_root(), "include"),
         SOURCE, ORACLE_C, "-L", lib_dir, "-lmoe_permute", "-L", cudart_dir, "-lcudart",
         f"-Wl,-rpath,{lib_dir}:{cudart_dir}", "-o", exe])
    return exe
