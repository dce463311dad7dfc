"""Device-side failure detection without a GPU fault.

The routing grid's blocks wait (bounded) for one another's histogram rows.
The debug build of the library (include/moe_permute_debug.h) makes every
block also wait for a table row that no block writes, with a 20 ms limit:
the waits must run out, set MOE_FLAG_BARRIER_TIMEOUT in the workspace status
word and return, leaving the context usable.  Nothing here faults, traps or
loops without bound.
"""
import time

import pytest
import torch

import moe_token_permute_gb300 as mp
from moe_token_permute_gb300 import _binding as b
from gpu_util import alloc_outputs, assert_metadata_equal, gpu_permute, oracle_route
from moe_token_permute_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

SHORT_WAIT_NS = 20_000_000  # 20 ms


@pytest.fixture
def debug_library(monkeypatch):
    """Route the package's calls through the debug build; restore the
    production wait afterwards."""
    dlib = b.debug_lib()
    monkeypatch.setattr(b, "_lib", dlib)
    yield dlib
    torch.cuda.synchronize()
    assert dlib.moe_debug_set_table_wait(0, b.TABLE_WAIT_NS) == b.MOE_OK


@pytest.mark.parametrize("name,T", [("mixtral", 4096), ("qwen3", 8192)])
def test_table_wait_runs_out_and_is_flagged(debug_library, name, T):
    inp = make_inputs(name, T, seed=7, with_rows=False)
    wl = inp["wl"]
    bufs = alloc_outputs(T, wl.K, wl.e_local, E=wl.E)
    ref = oracle_route(inp)

    # Production behaviour of the debug build first: exact, no flag.
    gpu_permute(inp, metadata_only=True, bufs=bufs)
    assert_metadata_equal(bufs, ref)
    assert mp.moe_read_status(bufs["ws"]) == 0

    # One row past the grid that nobody writes: every wait for it runs out.
    assert debug_library.moe_debug_set_table_wait(1, SHORT_WAIT_NS) == b.MOE_OK
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    gpu_permute(inp, metadata_only=True, bufs=bufs)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert mp.moe_read_status(bufs["ws"]) & b.MOE_FLAG_BARRIER_TIMEOUT
    assert elapsed < 1.0  # the 20 ms limit, not the 2 s production one

    # Back to the production wait: the context and the workspace still work.
    # The timed-out call advanced the table tag and cleared its extent, so
    # even without re-initialising the workspace the next call is exact.
    assert debug_library.moe_debug_set_table_wait(0, b.TABLE_WAIT_NS) == b.MOE_OK
    mp.moe_clear_status(bufs["ws"])
    gpu_permute(inp, metadata_only=True, bufs=bufs)
    assert_metadata_equal(bufs, ref)
    assert mp.moe_read_status(bufs["ws"]) == 0


@pytest.mark.parametrize("name,T", [("mixtral", 4096), ("dsv2lite", 8192)])
def test_table_wait_runs_out_with_row_copies_in_flight(debug_library, name, T):
    """The same forced timeout on a permute that also copies rows.  With an
    expert map (DeepSeek-V2-Lite) the single-launch kernel serves the call:
    its row loads are in flight into shared memory when its blocks give up,
    and its producer warp lets them land before the block exits.  Without one
    (Mixtral) the bulk-copy gather runs after a routing grid that gave up.
    Either way the flag is raised, nothing hangs, and the next call on the
    same workspace is exact."""
    from gpu_util import assert_rows_equal_full, oracle_full
    inp = make_inputs(name, T, seed=8, with_rows=False)
    wl = inp["wl"]
    bufs = alloc_outputs(T, wl.K, wl.e_local, wl.H, torch.bfloat16, E=wl.E)
    ref = oracle_full(inp)
    assert debug_library.moe_debug_set_table_wait(1, SHORT_WAIT_NS) == b.MOE_OK
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    gpu_permute(inp, bufs=bufs)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert mp.moe_read_status(bufs["ws"]) & b.MOE_FLAG_BARRIER_TIMEOUT
    assert elapsed < 1.0
    assert debug_library.moe_debug_set_table_wait(0, b.TABLE_WAIT_NS) == b.MOE_OK
    mp.moe_clear_status(bufs["ws"])
    gpu_permute(inp, bufs=bufs)
    assert_metadata_equal(bufs, ref)
    assert_rows_equal_full(inp, bufs, ref)
    assert mp.moe_read_status(bufs["ws"]) == 0
