"""The fp8 quantiser divides each element by its group's scale with an
fma-corrected reciprocal (Markstein's correction step) instead of an IEEE
division, where the scale lies in [2^-100, 2^100].  The debug build runs
every pair (x, amax) of finite bf16 values with |x| <= amax through both on
the GPU: the e4m3 codes must be identical for every pair, and the fp32
quotients wherever they are at least 2^-12 (smaller quotients all round to
the code 0 with x's sign).  The end-to-end bit-exactness against the CPU
oracle, which divides in IEEE arithmetic, is in tests/test_quant_gpu.py."""
import ctypes

import pytest

from moe_token_permute_gb300 import _binding as b
from moe_token_permute_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu


def test_division_matches_ieee_division_on_every_bf16_pair():
    cuda_build.build()
    counts = (ctypes.c_ulonglong * 4)()
    assert b.debug_lib().moe_debug_check_quant_division(counts) == b.MOE_OK
    checked, code_diff, quot_diff, outside = (int(c) for c in counts)
    # pairs of finite bf16 magnitudes with |x| <= amax, both signs of x and +-0
    assert checked > 1_000_000_000
    assert code_diff == 0
    assert quot_diff == 0
    assert outside < checked // 4  # the fast path covers the realistic range
