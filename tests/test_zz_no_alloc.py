"""moe_permute_noalloc: the permute entry point for callers that cannot
allocate device memory (for example a plugin whose host framework owns every
allocation, or a serving loop that must not call cudaMalloc once running).
It keeps its scratch in a static device array inside the library instead of
a caller workspace.  This test calls it through the C ABI several times in a
row, on different batches that share that array, and checks each result
against the CPU oracle (indices, offsets, every kept row and scale row, bit
for bit) and against moe_permute with a caller workspace.  It is collected
last and needs nothing from other tests."""
import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
import oracle
from gpu_util import assert_bytes_equal, bytes_of
from moe_token_permute_gb300 import _binding as b
from moe_token_permute_gb300 import build as cuda_build
from moe_token_permute_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

_DT = {torch.bfloat16: b.MOE_DTYPE_BF16, torch.float8_e4m3fn: b.MOE_DTYPE_FP8_E4M3}


def _p(t):
    return None if t is None else t.data_ptr()


def _outputs(wl, T, dtype, scale_cols):
    R = T * wl.K
    dev = "cuda"
    return dict(off=torch.full((wl.e_local + 1,), -5, dtype=torch.int64, device=dev),
                pidx=torch.full((R,), -5, dtype=torch.int32, device=dev),
                inv=torch.full((R,), -5, dtype=torch.int32, device=dev),
                ph=torch.zeros(R, wl.H, dtype=dtype, device=dev),
                ps=torch.zeros(R, scale_cols, dtype=torch.float32, device=dev) if scale_cols else None)


def _noalloc_call(inp, out):
    wl = inp["wl"]
    hidden = inp["hidden"]
    sc = inp["scales"]
    stream = torch.cuda.current_stream().cuda_stream
    return b.lib().moe_permute_noalloc(
        _p(hidden), _DT[hidden.dtype], _p(sc), 0 if sc is None else sc.shape[1],
        _p(inp["topk_ids"]), b.MOE_INDEX_INT32, _p(inp["expert_map"]),
        inp["T"], wl.H, wl.K, wl.E, wl.e_local,
        _p(out["ph"]), _p(out["ps"]), _p(out["off"]), _p(out["pidx"]), _p(out["inv"]), stream)


@pytest.fixture(scope="module", autouse=True)
def _library():
    cuda_build.build()
    b.lib()


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    # first: a large batch (cooperative path); second: a DeepSeek-V3-shaped
    # fp8 batch with scales and 256 experts; third: a small batch (single block)
    for name, T in (("mixtral", 3000), ("dsv3", 700), ("dsv2lite", 60)):
        inp = make_inputs(name, T, seed=11, device="cuda", with_rows=False)
        wl = inp["wl"]
        sc_cols = 0 if inp["scales"] is None else inp["scales"].shape[1]
        got = _outputs(wl, T, inp["hidden"].dtype, sc_cols)
        ref = _outputs(wl, T, inp["hidden"].dtype, sc_cols)
        assert _noalloc_call(inp, got) == b.MOE_OK
        ws = torch.empty(mp.moe_permute_workspace_size(T, wl.K, wl.E), dtype=torch.uint8,
                         device="cuda")
        mp.moe_permute_workspace_init(ws)
        mp.moe_permute(inp["hidden"], inp["topk_ids"], ref["off"], ref["pidx"], ref["inv"], ws,
                       num_experts=wl.E, num_local_experts=wl.e_local,
                       expert_map=inp["expert_map"], hidden_scales=inp["scales"],
                       permuted_hidden_states=ref["ph"], permuted_scales=ref["ps"])
        torch.cuda.synchronize()
        for k in ("off", "pidx", "inv"):
            assert torch.equal(got[k], ref[k]), (name, k)
        n = int(ref["off"][-1])
        assert torch.equal(got["ph"][:n].view(torch.uint8), ref["ph"][:n].view(torch.uint8))
        if sc_cols:
            assert torch.equal(got["ps"][:n], ref["ps"][:n])
        # and against the oracle itself
        orc = oracle.permute(inp["topk_ids"].cpu().numpy(), wl.E,
                             expert_map=None if inp["expert_map"] is None
                             else inp["expert_map"].cpu().numpy(),
                             E_local=wl.e_local, hidden=bytes_of(inp["hidden"]),
                             scales=None if inp["scales"] is None else inp["scales"].cpu().numpy())
        assert orc["flags"] == 0 and orc["n_valid"] == n
        np.testing.assert_array_equal(got["off"].cpu().numpy(), orc["offsets"])
        np.testing.assert_array_equal(got["pidx"].cpu().numpy(), orc["permuted_idx"])
        np.testing.assert_array_equal(got["inv"].cpu().numpy(), orc["inv_permuted_idx"])
        assert_bytes_equal(bytes_of(got["ph"][:n]), orc["permuted_hidden"][:n], name)
        if sc_cols:
            np.testing.assert_array_equal(got["ps"][:n].cpu().numpy().view(np.uint32),
                                          orc["permuted_scales"][:n].view(np.uint32))


def test_noalloc_empty_batch_with_many_experts():
    """T = 0 needs no histogram table: the offsets are zeroed whatever the
    expert count, and the call succeeds."""
    E = 1024
    off = torch.full((E + 1,), 9, dtype=torch.int64, device="cuda")
    rc = b.lib().moe_permute_noalloc(None, b.MOE_DTYPE_BF16, None, 0, None, b.MOE_INDEX_INT32,
                                     None, 0, 64, 8, E, E, None, None, off.data_ptr(), None, None,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == b.MOE_OK
    assert torch.count_nonzero(off).item() == 0


def test_noalloc_rejects_requests_beyond_its_scratch():
    T, K, E = 4096, 8, 1024  # needs more than the static array holds
    assert mp.moe_permute_workspace_size(T, K, E) > b.MOE_NOALLOC_SCRATCH_BYTES
    ids = torch.zeros(T, K, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int64, device="cuda")
    idx = torch.empty(T * K, dtype=torch.int32, device="cuda")
    rc = b.lib().moe_permute_noalloc(None, b.MOE_DTYPE_BF16, None, 0, ids.data_ptr(),
                                     b.MOE_INDEX_INT32, None, T, 1, K, E, E, None, None,
                                     off.data_ptr(), idx.data_ptr(), idx.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == b.MOE_ERR_WORKSPACE_TOO_SMALL
