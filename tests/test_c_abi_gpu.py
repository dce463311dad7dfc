"""A plain C program drives the C ABI on the GPU (device memory from the CUDA
runtime, no Python binding) and compares every output with the oracle bit for
bit: a single-launch batch, a routing-grid batch, and a batch with an expert
map and int64 ids."""
import subprocess

import pytest

from c_abi_build import build_consumer

pytestmark = pytest.mark.gpu


def test_c_program_matches_oracle(tmp_path):
    exe = build_consumer(str(tmp_path))
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("ok"), run.stdout
    assert "MISMATCH" not in run.stdout
