"""MoEPermuteScratch, the allocate-once wrapper (vLLM PR #43014 digest, "key
source excerpts": __post_init__, validate, token_expert_indices_view,
prepare_topk_ids; "implementation breakdown" item 5: two calls on one scratch
write the same storage with correct results), against the CPU oracle.

One scratch is built for the larger of two batches and driven with the larger
batch and then the smaller one, as a serving loop would.  Each call is compared
element by element with the oracle (offsets, both index maps, every kept row
and fp8 scale row, the unpermuted tokens), and every returned tensor must be a
view of the storage allocated at construction.  The two batch sizes straddle
the boundary between the single-launch kernel and the larger-batch paths.
"""
import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
import oracle
from gpu_util import (assert_bytes_equal, assert_unpermute_matches, bits16, bytes_of,
                      oracle_full)
from test_quant_gpu import bf16_rows
from moe_token_permute_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
G = mp._binding.MOE_QUANT_GROUP


def same_storage(view, base):
    """view starts at base's first element (the scratch hands out prefixes)."""
    return view.data_ptr() == base.data_ptr()


def check_permute_result(res, scratch, inp, ref):
    n = ref["n_valid"]
    R = inp["T"] * inp["wl"].K
    np.testing.assert_array_equal(res["expert_first_token_offset"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(res["permuted_idx"].cpu().numpy(), ref["permuted_idx"])
    np.testing.assert_array_equal(res["inv_permuted_idx"].cpu().numpy(), ref["inv_permuted_idx"])
    assert res["permuted_idx"].numel() == R and res["inv_permuted_idx"].numel() == R
    assert same_storage(res["expert_first_token_offset"], scratch.expert_first_token_offset)
    assert same_storage(res["permuted_idx"], scratch.permuted_idx)
    assert same_storage(res["inv_permuted_idx"], scratch.inv_permuted_idx)
    assert same_storage(res["permuted_hidden_states"], scratch.permuted_hidden_states)
    assert_bytes_equal(bytes_of(res["permuted_hidden_states"][:n]), ref["permuted_hidden"][:n],
                       "permuted_hidden_states")
    if ref["permuted_scales"] is not None:
        assert same_storage(res["permuted_scales"], scratch.permuted_scales)
        np.testing.assert_array_equal(res["permuted_scales"][:n].cpu().numpy().view(np.uint32),
                                      ref["permuted_scales"][:n].view(np.uint32))


# (workload, larger T, smaller T, id dtype): the larger batch takes the routing
# grid and the gather, the smaller one the single-launch kernel.
CASES = [("dsv2lite", 1000, 300, torch.int32),   # expert map: 16 of 64 experts local
         ("dsv3", 600, 200, torch.int32),        # fp8 rows with [T, 56] scales
         ("qwen3", 2000, 200, torch.int64),      # Zipf routing, int64 ids
         ("mixtral", 3000, 1000, torch.int64)]


@pytest.mark.parametrize("name,T_big,T_small,idt", CASES,
                         ids=[f"{c[0]}-T{c[1]}-T{c[2]}-{str(c[3])[6:]}" for c in CASES])
def test_scratch_permute_unpermute_match_oracle(name, T_big, T_small, idt):
    wl = WORKLOADS[name]
    probe = make_inputs(name, 1, seed=0, with_rows=False)
    sc_cols = 0 if probe["scales"] is None else probe["scales"].shape[1]
    scratch = mp.MoEPermuteScratch(T_big, wl.K, wl.E, wl.e_local, DEV, wl.H,
                                   probe["hidden"].dtype, scale_cols=sc_cols)
    storage = {k: getattr(scratch, k).data_ptr()
               for k in ("workspace", "expert_first_token_offset", "permuted_idx",
                         "inv_permuted_idx", "permuted_hidden_states", "unpermuted")}
    for T in (T_big, T_small):
        inp = make_inputs(name, T, seed=T)
        ref = oracle_full(inp)
        assert ref["flags"] == 0
        emap = None if inp["expert_map"] is None else inp["expert_map"].to(DEV)
        ids = inp["topk_ids"].to(device=DEV, dtype=idt)
        assert scratch.prepare_topk_ids(ids) is ids
        res = scratch.permute(inp["hidden"].to(DEV), ids, expert_map=emap,
                              hidden_scales=None if inp["scales"] is None
                              else inp["scales"].to(DEV))
        check_permute_result(res, scratch, inp, ref)
        # unpermute through the scratch's inverse map, into its own buffer
        out = scratch.unpermute(inp["rows"].to(DEV), inp["topk_weights"].to(DEV))
        assert out.shape == (T, wl.H) and same_storage(out, scratch.unpermuted)
        ref_out, flags = oracle.unpermute(bits16(inp["rows"]), inp["topk_weights"].numpy(),
                                          ref["inv_permuted_idx"])
        assert flags == 0
        assert_unpermute_matches(bits16(out), ref_out)
        # and into a caller buffer
        mine = torch.empty(T, wl.H, dtype=torch.bfloat16, device=DEV)
        assert scratch.unpermute(inp["rows"].to(DEV), inp["topk_weights"].to(DEV), out=mine) is mine
        assert_unpermute_matches(bits16(mine), ref_out)
        assert scratch.read_status() == 0
    # no call replaced a buffer
    for k, ptr in storage.items():
        assert getattr(scratch, k).data_ptr() == ptr, k


@pytest.mark.parametrize("T_big,T_small", [(600, 100)])
def test_scratch_quant_fp8_matches_oracle(T_big, T_small):
    """bf16 rows quantised to fp8 e4m3 plus per-128-column scales on the way
    into the scratch (DeepSeek-V3 shape), against the oracle's quantiser and
    permute."""
    wl = WORKLOADS["dsv3"]
    scratch = mp.MoEPermuteScratch(T_big, wl.K, wl.E, wl.e_local, DEV, wl.H,
                                   torch.float8_e4m3fn, scale_cols=wl.H // G)
    for T in (T_big, T_small):
        inp = make_inputs("dsv3", T, seed=T + 1, with_rows=False)
        hidden = bf16_rows(T, wl.H, seed=T + 2)
        q, s = oracle.quantize_fp8(bits16(hidden), G)
        ref = oracle.permute(inp["topk_ids"].numpy(), wl.E, hidden=q, scales=s)
        res = scratch.permute_quant_fp8(hidden.to(DEV), inp["topk_ids"].to(DEV))
        check_permute_result(res, scratch, inp, ref)


def test_scratch_batched_matches_oracle():
    """Batched [E_local, M, H] layout through the scratch, capacity overflow
    included (Qwen3 shape, Zipf routing), then unpermute over the batched
    rows through the slot map."""
    wl = WORKLOADS["qwen3"]
    T, M = 1500, 64
    scratch = mp.MoEPermuteScratch(T, wl.K, wl.E, wl.e_local, DEV, wl.H, torch.bfloat16,
                                   max_rows_per_expert=M)
    inp = make_inputs("qwen3", T, seed=21, with_rows=False)
    ref = oracle.permute_batched(inp["topk_ids"].numpy(), wl.E, M, hidden=bytes_of(inp["hidden"]))
    assert ref["flags"] == mp.MOE_FLAG_CAPACITY_OVERFLOW
    res = scratch.permute_batched(inp["hidden"].to(DEV), inp["topk_ids"].to(DEV))
    np.testing.assert_array_equal(res["expert_num_tokens"].cpu().numpy(), ref["expert_num_tokens"])
    np.testing.assert_array_equal(res["inv_permuted_idx"].cpu().numpy(), ref["inv_permuted_idx"])
    assert same_storage(res["batched_hidden_states"], scratch.batched_hidden_states)
    assert res["batched_hidden_states"].shape == (wl.e_local, M, wl.H)
    slots = np.concatenate([e * M + np.arange(c) for e, c in enumerate(ref["expert_num_tokens"])])
    got_rows = bytes_of(scratch.batched_hidden_states[torch.from_numpy(slots).to(DEV)])
    assert_bytes_equal(got_rows, ref["batched_hidden"][slots], "batched_hidden_states")
    assert scratch.read_status() == mp.MOE_FLAG_CAPACITY_OVERFLOW
    scratch.clear_status()
    g = torch.Generator().manual_seed(5)
    rows = torch.randn(wl.e_local * M, wl.H, generator=g).to(torch.bfloat16)
    out = scratch.unpermute(rows.to(DEV), inp["topk_weights"].to(DEV))
    ref_out, flags = oracle.unpermute(bits16(rows), inp["topk_weights"].numpy(),
                                      ref["inv_permuted_idx"])
    assert flags == 0
    assert_unpermute_matches(bits16(out), ref_out)
    assert scratch.read_status() == 0


def test_scratch_token_expert_indices_view_and_validate():
    scratch = mp.MoEPermuteScratch(64, 6, 64, 16, DEV, 256, torch.bfloat16)
    v = scratch.token_expert_indices_view(10)
    assert v.shape == (10, 6) and v.dtype == torch.int32
    assert same_storage(v, scratch.token_expert_indices)
    assert torch.equal(v.cpu(), torch.arange(60, dtype=torch.int32).view(10, 6))
    ids = torch.zeros(65, 6, dtype=torch.int32, device=DEV)
    hid = torch.zeros(65, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):  # more tokens than the scratch holds
        scratch.permute(hid, ids)
    with pytest.raises(ValueError):  # wrong top-k
        scratch.permute(hid[:8], torch.zeros(8, 5, dtype=torch.int32, device=DEV))
    with pytest.raises(ValueError):  # wrong hidden size
        scratch.permute(torch.zeros(8, 128, dtype=torch.bfloat16, device=DEV), ids[:8])
    with pytest.raises(ValueError):  # wrong dtype
        scratch.permute(hid[:8].float(), ids[:8])
    with pytest.raises(ValueError):  # ids on the host
        scratch.permute(hid[:8], ids[:8].cpu())
    with pytest.raises(ValueError):  # no batched buffers in this scratch
        scratch.permute_batched(hid[:8], ids[:8])
    with pytest.raises(ValueError):  # not an fp8 scratch
        scratch.permute_quant_fp8(hid[:8], ids[:8])
