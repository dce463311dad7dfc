"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every workload shape the library is measured on, at every token count of its
sweep, compared element by element: offsets, both index maps, every kept
permuted row (and fp8 scale row) and every unpermuted token.  Up to 4096
tokens the inputs are drawn on the host; above that they are drawn on the
device (the largest case, DeepSeek-V3 at 32768 tokens, moves 1.9 GB of rows)
and copied back for the oracle, which computes the whole problem.
Bar: bit-exact indices, offsets, rows and scales; unpermute within
2^-7*|ref| + 1e-6 of the oracle (and in fact bit-identical).
"""
import pytest
import torch

import oracle
import pins
from gpu_util import (assert_metadata_equal, assert_rows_equal_full, assert_unpermute_matches,
                      bits16, gpu_permute, gpu_unpermute, oracle_full)
from moe_token_permute_gb300 import moe_read_status
from moe_token_permute_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

FULL_MAX_T = 4096
FULL = [(n, T) for n, wl in WORKLOADS.items() for T in wl.T_sweep if T <= FULL_MAX_T]
LARGE = [(n, T) for n, wl in WORKLOADS.items() for T in wl.T_sweep if T > FULL_MAX_T]


@pytest.mark.parametrize("name,T", FULL, ids=[f"{n}-T{T}" for n, T in FULL])
def test_full_parity(name, T):
    inp = make_inputs(name, T, seed=0)
    wl = inp["wl"]
    ref = oracle_full(inp)
    assert ref["flags"] == 0
    bufs = gpu_permute(inp)
    assert_metadata_equal(bufs, ref)
    assert_rows_equal_full(inp, bufs, ref)
    assert moe_read_status(bufs["ws"]) == 0
    pins.check_routing_invariants(inp["topk_ids"].numpy(), wl.E,
                                  dict(offsets=bufs["offsets"].cpu().numpy(),
                                       permuted_idx=bufs["pidx"].cpu().numpy(),
                                       inv_permuted_idx=bufs["inv"].cpu().numpy()),
                                  None if inp["expert_map"] is None else inp["expert_map"].numpy(),
                                  wl.e_local)
    # int64 ids give the same result
    bufs64 = gpu_permute(inp, ids_dtype=torch.int64)
    assert_metadata_equal(bufs64, ref)
    assert_rows_equal_full(inp, bufs64, ref)
    # unpermute on the oracle's inverse map
    out = gpu_unpermute(inp["rows"], inp["topk_weights"],
                        torch.from_numpy(ref["inv_permuted_idx"]), ws=bufs["ws"])
    ref_out, flags = oracle.unpermute(bits16(inp["rows"]), inp["topk_weights"].numpy(),
                                      ref["inv_permuted_idx"])
    assert flags == 0
    assert_unpermute_matches(bits16(out), ref_out)
    assert moe_read_status(bufs["ws"]) == 0


@pytest.mark.parametrize("name,T", LARGE, ids=[f"{n}-T{T}" for n, T in LARGE])
def test_large_full(name, T):
    inp = make_inputs(name, T, seed=0, device="cuda")
    wl = inp["wl"]
    ref = oracle_full(inp)
    assert ref["flags"] == 0
    bufs = gpu_permute(inp)
    assert_metadata_equal(bufs, ref)
    assert_rows_equal_full(inp, bufs, ref)
    assert moe_read_status(bufs["ws"]) == 0
    pins.check_routing_invariants(inp["topk_ids"].cpu().numpy(), wl.E,
                                  dict(offsets=bufs["offsets"].cpu().numpy(),
                                       permuted_idx=bufs["pidx"].cpu().numpy(),
                                       inv_permuted_idx=bufs["inv"].cpu().numpy()),
                                  None if inp["expert_map"] is None
                                  else inp["expert_map"].cpu().numpy(), wl.e_local)
    del ref["permuted_hidden"], bufs["ph"]
    # unpermute of every token, on the inverse map the GPU wrote (equal to the
    # oracle's, checked above), against the oracle over all T*K rows
    out = gpu_unpermute(inp["rows"], inp["topk_weights"], bufs["inv"], ws=bufs["ws"])
    ref_out, flags = oracle.unpermute(bits16(inp["rows"]), inp["topk_weights"].cpu().numpy(),
                                      ref["inv_permuted_idx"])
    assert flags == 0
    assert_unpermute_matches(bits16(out), ref_out)
    assert moe_read_status(bufs["ws"]) == 0
