"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every workload shape the library is measured on, at every token count of its
sweep.  Up to 4096 tokens the whole output is compared with the oracle; at the
largest token counts (inputs drawn on the device) the routing metadata is still
compared in full, the row copy is checked as a property over all rows and
against the oracle on sampled rows, and unpermute is compared on sampled tokens.
Bar: bit-exact indices, offsets, rows and scales; unpermute within
2^-7*|ref| + 1e-6 of the oracle (and in fact bit-identical).
"""
import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_util import (assert_metadata_equal, assert_rows_equal_full, assert_unpermute_matches,
                      bits16, bytes_of, gpu_permute, gpu_unpermute, oracle_full, oracle_route)
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
def test_large_sampled(name, T):
    inp = make_inputs(name, T, seed=0, device="cuda")
    wl = inp["wl"]
    K = wl.K
    ref = oracle_route(inp)
    bufs = gpu_permute(inp)
    assert_metadata_equal(bufs, ref)
    assert moe_read_status(bufs["ws"]) == 0
    n = ref["n_valid"]
    pidx = bufs["pidx"][:n].long()
    # row-copy property over every row, evaluated on the device
    src = pidx // K
    hid = inp["hidden"].view(torch.uint8) if inp["hidden"].element_size() == 1 else inp["hidden"].view(torch.int16)
    assert torch.equal(bufs["ph"][:n].view(hid.dtype), hid[src])
    if bufs["ps"] is not None:
        assert torch.equal(bufs["ps"][:n], inp["scales"][src])
    # sampled rows against the oracle's routing and the host copy of hidden
    g = np.random.default_rng(1)
    ps = np.unique(np.concatenate([[0, n - 1], g.integers(0, n, 64)]))
    host_hidden = bytes_of(inp["hidden"])
    got = bytes_of(bufs["ph"][torch.from_numpy(ps).cuda()])
    np.testing.assert_array_equal(got, host_hidden[ref["permuted_idx"][ps] // K])
    # unpermute on sampled tokens, oracle on the compacted sub-problem
    inv = torch.from_numpy(ref["inv_permuted_idx"]).cuda()
    out = gpu_unpermute(inp["rows"], inp["topk_weights"], inv, ws=bufs["ws"])
    ts = np.unique(np.concatenate([[0, T - 1], g.integers(0, T, 48)]))
    inv_s = ref["inv_permuted_idx"].reshape(T, K)[ts]
    rows_s = bits16(inp["rows"][torch.from_numpy(np.maximum(inv_s, 0).reshape(-1)).cuda()])
    inv_c = np.where(inv_s >= 0, np.arange(inv_s.size).reshape(inv_s.shape), -1).astype(np.int32)
    ref_out, _ = oracle.unpermute(rows_s, inp["topk_weights"].cpu().numpy()[ts], inv_c.reshape(-1))
    assert_unpermute_matches(bits16(out[torch.from_numpy(ts).cuda()]), ref_out)
    assert moe_read_status(bufs["ws"]) == 0
