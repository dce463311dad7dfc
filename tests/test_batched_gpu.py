"""GPU parity of the batched activation layout (moe_permute_batched) against
the CPU oracle's batched permute: per-expert counts, the slot map and every
filled slot's row (and scale row) must match bit for bit, with and without
capacity overflow; unpermute over the batched rows must match the oracle."""
import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
import oracle
from gpu_util import assert_unpermute_matches, bits16, bytes_of
from moe_token_permute_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


def run_batched(inp, M, metadata_only=False, ids_dtype=torch.int32):
    wl = inp["wl"]
    T = inp["T"]
    dev = "cuda"
    counts = torch.full((wl.e_local,), -3, dtype=torch.int32, device=dev)
    inv = torch.full((T * wl.K,), -3, dtype=torch.int32, device=dev)
    ws = torch.empty(mp.moe_permute_workspace_size(T, wl.K, wl.E), dtype=torch.uint8, device=dev)
    mp.moe_permute_workspace_init(ws)
    hidden = inp["hidden"].to(dev)
    scales = None if inp["scales"] is None else inp["scales"].to(dev)
    bh = bs = None
    if not metadata_only:
        bh = torch.zeros(wl.e_local * M, wl.H, dtype=hidden.dtype, device=dev)
        if scales is not None:
            bs = torch.zeros(wl.e_local * M, scales.shape[1], dtype=torch.float32, device=dev)
    mp.moe_permute_batched(None if metadata_only else hidden,
                           inp["topk_ids"].to(device=dev, dtype=ids_dtype), counts, inv, ws,
                           num_experts=wl.E, num_local_experts=wl.e_local, max_rows_per_expert=M,
                           expert_map=None if inp["expert_map"] is None else inp["expert_map"].to(dev),
                           hidden_scales=None if metadata_only else scales,
                           batched_hidden_states=bh, batched_scales=bs)
    return dict(counts=counts, inv=inv, bh=bh, bs=bs, ws=ws)


def oracle_batched(inp, M):
    wl = inp["wl"]
    return oracle.permute_batched(
        inp["topk_ids"].cpu().numpy(), wl.E, M,
        expert_map=None if inp["expert_map"] is None else inp["expert_map"].cpu().numpy(),
        E_local=wl.e_local, hidden=bytes_of(inp["hidden"]),
        scales=None if inp["scales"] is None else inp["scales"].cpu().numpy())


def filled_slots(counts, M):
    return np.concatenate([e * M + np.arange(c) for e, c in enumerate(counts)]).astype(np.int64)


def check(M, got, ref, expect_flags):
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), ref["expert_num_tokens"])
    np.testing.assert_array_equal(got["inv"].cpu().numpy(), ref["inv_permuted_idx"])
    assert ref["flags"] == expect_flags
    assert mp.moe_read_status(got["ws"]) == expect_flags
    if got["bh"] is not None:
        slots = filled_slots(ref["expert_num_tokens"], M)
        idx = torch.from_numpy(slots).cuda()
        np.testing.assert_array_equal(bytes_of(got["bh"][idx]), ref["batched_hidden"][slots])
        if got["bs"] is not None:
            np.testing.assert_array_equal(got["bs"][idx].cpu().numpy(), ref["batched_scales"][slots])


CASES = [("mixtral", 4096, None), ("qwen3", 1024, None), ("dsv2lite", 256, None),
         ("dsv3", 128, None), ("tiny", 16, None), ("qwen3", 64, 8), ("dsv3", 300, 12)]


@pytest.mark.parametrize("name,T,M", CASES, ids=[f"{n}-T{T}-M{M}" for n, T, M in CASES])
def test_batched_matches_oracle(name, T, M):
    inp = make_inputs(name, T, seed=3)
    if M is None:
        M = T  # distinct experts per token: an expert gets at most T rows
    ref = oracle_batched(inp, M)
    got = run_batched(inp, M)
    check(M, got, ref, ref["flags"])
    if M == T:
        assert ref["flags"] == 0


def test_batched_capacity_overflow_is_flagged():
    inp = make_inputs("qwen3", 512, seed=4)  # Zipf routing: popular experts overflow
    ref = oracle_batched(inp, 16)
    assert ref["flags"] == mp.MOE_FLAG_CAPACITY_OVERFLOW
    got = run_batched(inp, 16, ids_dtype=torch.int64)
    check(16, got, ref, mp.MOE_FLAG_CAPACITY_OVERFLOW)


def test_batched_metadata_only_large():
    inp = make_inputs("qwen3", 16384, seed=5, device="cuda", with_rows=False)
    M = 16384
    wl = inp["wl"]
    got = run_batched(inp, M, metadata_only=True)
    ref = oracle.permute_batched(inp["topk_ids"].cpu().numpy(), wl.E, M)
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), ref["expert_num_tokens"])
    np.testing.assert_array_equal(got["inv"].cpu().numpy(), ref["inv_permuted_idx"])


def test_unpermute_over_batched_rows():
    """The batched GEMM output reduces back to tokens through the slot map."""
    inp = make_inputs("dsv2lite", 1000, seed=6)
    wl = inp["wl"]
    M = 1000
    got = run_batched(inp, M, metadata_only=True)
    g = torch.Generator().manual_seed(9)
    rows = torch.randn(wl.e_local * M, wl.H, generator=g).to(torch.bfloat16)
    out = torch.empty(1000, wl.H, dtype=torch.bfloat16, device="cuda")
    mp.moe_unpermute(rows.cuda(), inp["topk_weights"].cuda(), got["inv"], out)
    ref_out, _ = oracle.unpermute(bits16(rows), inp["topk_weights"].numpy(),
                                  got["inv"].cpu().numpy())
    assert_unpermute_matches(bits16(out), ref_out)


def test_batched_zero_tokens():
    inp = make_inputs("qwen3", 0, seed=1, with_rows=False)
    got = run_batched(inp, 4, metadata_only=True)
    assert got["counts"].cpu().tolist() == [0] * inp["wl"].E


def test_batched_metadata_only_large_table():
    """256 local experts at T = 20000: the routing grid's histogram table would
    reach 152 x 256 entries, so it runs rounds of 8 rows per lane over half the
    blocks; the batched slot map and counts must still match the oracle."""
    inp = make_inputs("dsv3", 20000, seed=8, with_rows=False)
    wl = inp["wl"]
    M = 512  # popular experts overflow: rows past the capacity are dropped and flagged
    got = run_batched(inp, M, metadata_only=True)
    ref = oracle.permute_batched(inp["topk_ids"].cpu().numpy(), wl.E, M)
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), ref["expert_num_tokens"])
    np.testing.assert_array_equal(got["inv"].cpu().numpy(), ref["inv_permuted_idx"])
    assert mp.moe_read_status(got["ws"]) == ref["flags"]
