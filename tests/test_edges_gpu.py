"""GPU edge cases against the oracle: empty and ragged inputs, the maximum
sizes the API accepts, the single-launch / multi-launch boundary, vector-width
fallbacks and misaligned pointers, dropped and invalid ids, the status word,
scratch reuse and CUDA-graph capture."""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
import oracle
from gpu_util import (alloc_outputs, assert_metadata_equal, assert_rows_equal_full,
                      assert_unpermute_matches, bits16, gpu_permute, gpu_unpermute, oracle_full)

pytestmark = pytest.mark.gpu

CHUNK = 8192  # sizes around the rows one block ranks in one pass (single launch: <= 2048 rows)


def custom_inputs(T, K, E, H, dtype=torch.bfloat16, E_local=None, emap=None, ids=None,
                  scale_cols=0, seed=0, id_range=None, misalign=0):
    g = torch.Generator().manual_seed(seed)
    if ids is None:
        lo, hi = id_range if id_range is not None else (0, E)
        ids = torch.randint(lo, hi, (T, K), generator=g, dtype=torch.int32)
    if dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        raw = torch.randint(0, 256, (T * H + misalign,), generator=g, dtype=torch.uint8)
        flat = raw.view(dtype)
    else:
        flat = torch.randn(T * H + misalign, generator=g).to(dtype)
    hidden = flat[misalign:].view(T, H) if T * H else flat[:0].view(T, H)
    scales = torch.rand(T, scale_cols, generator=g) if scale_cols else None
    weights = torch.rand(T, K, generator=g)
    rows = torch.randn(T * K, H, generator=g).to(torch.bfloat16)
    wl = SimpleNamespace(H=H, E=E, K=K, e_local=E if E_local is None else E_local)
    return dict(wl=wl, T=T, hidden=hidden, scales=scales, topk_ids=ids, topk_weights=weights,
                rows=rows, expert_map=emap)


def to_device_keep_offset(t, misalign):
    """Copy to the GPU keeping a misalignment of `misalign` elements."""
    if t is None:
        return None
    flat = torch.empty(t.numel() + misalign, dtype=t.dtype, device="cuda")
    dst = flat[misalign:].view(t.shape)
    dst.copy_(t)
    return dst


def check_case(inp, expect_flags=0, unpermute=True, ids_dtype=torch.int32):
    ref = oracle_full(inp)
    assert ref["flags"] == expect_flags
    bufs = gpu_permute(inp, ids_dtype=ids_dtype)
    assert_metadata_equal(bufs, ref)
    assert_rows_equal_full(inp, bufs, ref)
    assert mp.moe_read_status(bufs["ws"]) == expect_flags
    if unpermute and inp["T"] > 0:
        out = gpu_unpermute(inp["rows"], inp["topk_weights"],
                            torch.from_numpy(ref["inv_permuted_idx"]))
        ref_out, _ = oracle.unpermute(bits16(inp["rows"]), inp["topk_weights"].numpy(),
                                      ref["inv_permuted_idx"])
        assert_unpermute_matches(bits16(out), ref_out)
    return ref, bufs


def test_zero_tokens():
    inp = custom_inputs(0, 4, 16, 64)
    bufs = gpu_permute(inp)
    assert bufs["offsets"].cpu().tolist() == [0] * 17
    out = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    mp.moe_unpermute(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"),
                     torch.empty(0, 4, device="cuda"),
                     torch.empty(0, dtype=torch.int32, device="cuda"), out)


@pytest.mark.parametrize("T,K", [(2048, 1), (2049, 1), (256, 8), (257, 8),
                                 (3072, 1), (3073, 1), (384, 8), (385, 8),
                                 (CHUNK, 1), (CHUNK + 1, 1), (1024, 8), (1025, 8),
                                 (3 * CHUNK // 2 + 3, 2), (5 * CHUNK + 17, 1)])
def test_single_and_multi_launch_boundary(T, K):
    """Around 2048 rows (one block ranks 2 rows per lane, then 4), 3072 (the
    single launch ends without a map) and the routing grid's round sizes."""
    check_case(custom_inputs(T, K, 64, 96, seed=T))


@pytest.mark.parametrize("T,K", [(2048, 2), (2049, 2), (4096, 1), (4097, 1), (512, 8), (513, 8)])
def test_single_launch_boundary_with_expert_map(T, K):
    """With an expert map the single launch serves up to 4096 rows, and the
    single-launch expert-map kernel takes over above."""
    g = torch.Generator().manual_seed(T + K)
    emap = torch.full((64,), -1, dtype=torch.int32)
    emap[torch.randperm(64, generator=g)[:16]] = torch.randperm(16, generator=g).to(torch.int32)
    check_case(custom_inputs(T, K, 64, 128, E_local=16, emap=emap, seed=T + K))


@pytest.mark.parametrize("H,dtype", [(1, torch.bfloat16), (3, torch.bfloat16),
                                     (7, torch.bfloat16), (100, torch.bfloat16),
                                     (129, torch.float16), (5, torch.float8_e4m3fn),
                                     (24, torch.float8_e5m2), (33, torch.float32)])
@pytest.mark.parametrize("T", [37, 2500])
def test_row_widths(H, dtype, T):
    check_case(custom_inputs(T, 4, 8, H, dtype=dtype, seed=H))


@pytest.mark.parametrize("misalign", [1, 2, 3])
@pytest.mark.parametrize("T", [50, 3000])
def test_misaligned_rows(misalign, T):
    H, K, E = 256, 3, 16
    inp = custom_inputs(T, K, E, H, seed=misalign)
    ref = oracle_full(inp)
    hidden = to_device_keep_offset(inp["hidden"], misalign)
    ids = inp["topk_ids"].cuda()
    bufs = alloc_outputs(T, K, E, None, None)
    ph_flat = torch.zeros(T * K * H + misalign, dtype=torch.bfloat16, device="cuda")
    ph = ph_flat[misalign:].view(T * K, H)
    mp.moe_permute(hidden, ids, bufs["offsets"], bufs["pidx"], bufs["inv"], bufs["ws"],
                   num_experts=E, permuted_hidden_states=ph)
    assert_metadata_equal(bufs, ref)
    n = ref["n_valid"]
    np.testing.assert_array_equal(bits16(ph[:n]), ref["permuted_hidden"][:n].view(np.uint16))
    rows = to_device_keep_offset(inp["rows"], misalign)
    out_flat = torch.zeros(T * H + misalign, dtype=torch.bfloat16, device="cuda")
    out = out_flat[misalign:].view(T, H)
    mp.moe_unpermute(rows, inp["topk_weights"].cuda(), bufs["inv"], out)
    ref_out, _ = oracle.unpermute(bits16(inp["rows"]), inp["topk_weights"].numpy(),
                                  ref["inv_permuted_idx"])
    assert_unpermute_matches(bits16(out), ref_out)


@pytest.mark.parametrize("T", [300, 20000])
def test_max_topk_and_max_local_experts(T):
    K = mp.MOE_MAX_TOPK if T == 300 else 8
    E = mp.MOE_MAX_LOCAL_EXPERTS
    check_case(custom_inputs(T, K, E, 64, seed=5))


@pytest.mark.parametrize("T,K", [(256, 8), (2048, 1), (1, 32), (384, 8)])
def test_single_launch_with_max_local_experts(T, K):
    """Up to 3072 rows over 1024 experts in one launch: every warp ranks (2 or
    4 rows per lane), and the per-warp counts take up to [32][1024] ints of
    shared memory."""
    check_case(custom_inputs(T, K, mp.MOE_MAX_LOCAL_EXPERTS, 64, seed=T + K))


@pytest.mark.parametrize("T", [682, 700, 9000])
def test_expert_map_with_max_local_experts(T):
    """1024 local experts of 2048 through an expert map: one launch of the
    small-batch kernel at 4092 rows, the expert-map kernel above."""
    E, EL = 2048, 1024
    g = torch.Generator().manual_seed(3)
    emap = torch.full((E,), -1, dtype=torch.int32)
    chosen = torch.randperm(E, generator=g)[:EL]
    emap[chosen] = torch.randperm(EL, generator=g).to(torch.int32)
    inp = custom_inputs(T, 6, E, 64, E_local=EL, emap=emap, seed=4)
    check_case(inp)


@pytest.mark.parametrize("T", [40, 4000])
def test_invalid_ids_are_dropped_and_flagged(T):
    inp = custom_inputs(T, 4, 8, 32, id_range=(-2, 10), seed=9)
    check_case(inp, expect_flags=mp.MOE_FLAG_ID_OUT_OF_RANGE)
    check_case(inp, expect_flags=mp.MOE_FLAG_ID_OUT_OF_RANGE, ids_dtype=torch.int64)


@pytest.mark.parametrize("T", [40, 4000])
def test_bad_map_values_are_dropped_and_flagged(T):
    emap = torch.tensor([0, -1, 1, 7, -3, 2, -1, 3], dtype=torch.int32)
    inp = custom_inputs(T, 3, 8, 32, E_local=4, emap=emap, seed=10)
    check_case(inp, expect_flags=mp.MOE_FLAG_MAP_OUT_OF_RANGE)


@pytest.mark.parametrize("T", [9, 5000])
def test_duplicate_experts_and_single_expert(T):
    ids = torch.full((T, 4), 3, dtype=torch.int32)
    ids[::2, 1] = 0
    check_case(custom_inputs(T, 4, 6, 40, ids=ids))


@pytest.mark.parametrize("T", [1, 2, 31])
def test_every_row_dropped(T):
    emap = torch.full((8,), -1, dtype=torch.int32)
    emap[7] = 0
    ids = torch.zeros(T, 2, dtype=torch.int32)
    ref, bufs = check_case(custom_inputs(T, 2, 8, 16, E_local=1, emap=emap, ids=ids))
    assert ref["n_valid"] == 0
    out = gpu_unpermute(torch.randn(2 * T, 16).to(torch.bfloat16), torch.rand(T, 2),
                        torch.from_numpy(ref["inv_permuted_idx"]))
    assert torch.all(bits16_t(out) == 0)  # +0.0 exactly


def bits16_t(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("T", [64, 6000])
def test_metadata_only(T):
    inp = custom_inputs(T, 6, 32, 64, seed=11)
    ref = oracle_full(inp)
    bufs = gpu_permute(inp, metadata_only=True)
    assert_metadata_equal(bufs, ref)


@pytest.mark.parametrize("T", [64, 6000])
def test_fp8_scales_odd_width(T):
    inp = custom_inputs(T, 4, 16, 384, dtype=torch.float8_e4m3fn, scale_cols=3, seed=12)
    check_case(inp)


@pytest.mark.parametrize("bad", [{5: "end"}, {11: -4}, {5: "end", 11: -4}, {3: -1}],
                         ids=["past_end", "below_minus_one", "both", "minus_one_only"])
def test_unpermute_flags_bad_inverse_indices(bad):
    """An inverse index outside [-1, num_rows) names no row: it is skipped and
    raises MOE_FLAG_INV_OUT_OF_RANGE; -1 is a dropped row and raises nothing.
    The status word must equal the oracle's flags on the raw map."""
    T, K, H = 20, 3, 48
    rows = torch.randn(T * K, H).to(torch.bfloat16)
    w = torch.rand(T, K)
    inv = torch.randperm(T * K).to(torch.int32)
    for i, v in bad.items():
        inv[i] = T * K if v == "end" else v
    ws = torch.empty(mp.moe_permute_workspace_size(T, K, 4), dtype=torch.uint8, device="cuda")
    mp.moe_permute_workspace_init(ws)
    out = gpu_unpermute(rows, w, inv, ws=ws)
    ref_out, flags = oracle.unpermute(bits16(rows), w.numpy(), inv.numpy())
    assert mp.moe_read_status(ws) == flags
    assert flags == (0 if bad == {3: -1} else oracle.FLAG_INV_RANGE)
    assert_unpermute_matches(bits16(out), ref_out)
    mp.moe_clear_status(ws)
    assert mp.moe_read_status(ws) == 0


@pytest.mark.parametrize("T", [100, 7000])
def test_scratch_reuse_two_calls(T):
    """Two calls on one scratch write the same buffers with identical results
    (vLLM PR #43014 digest, test and benchmark item: reuse of the scratch)."""
    from moe_token_permute_gb300.workloads import make_inputs
    inp = make_inputs("qwen3", T, seed=2)
    wl = inp["wl"]
    hidden = inp["hidden"].cuda()
    ids = inp["topk_ids"].cuda()
    scratch = mp.MoEPermuteScratch(T, wl.K, wl.E, wl.E, torch.device("cuda"), wl.H, hidden.dtype)
    a = scratch.permute(hidden, ids)
    snap = {k: v.clone() for k, v in a.items() if v is not None}
    ptrs = {k: v.data_ptr() for k, v in a.items() if v is not None}
    b = scratch.permute(hidden, ids)
    for k, v in b.items():
        if v is None:
            continue
        assert v.data_ptr() == ptrs[k]
        assert torch.equal(v, snap[k])


@pytest.mark.parametrize("T", [100, 7000])
def test_poisoned_workspace_after_init(T):
    from moe_token_permute_gb300.workloads import make_inputs
    inp = make_inputs("dsv2lite", T, seed=3)
    ref = oracle_full(inp)
    wl = inp["wl"]
    bufs = alloc_outputs(T, wl.K, wl.e_local, wl.H, torch.bfloat16, E=wl.E)
    bufs["ws"].fill_(0xFF)
    mp.moe_permute_workspace_init(bufs["ws"])
    gpu_permute(inp, bufs=bufs)
    assert_metadata_equal(bufs, ref)
    assert_rows_equal_full(inp, bufs, ref)


@pytest.mark.parametrize("T", [100, 7000])
def test_cuda_graph_capture(T):
    """permute + unpermute capture into a CUDA graph (no allocation, no host
    sync inside the calls) and the replay reproduces the eager result."""
    from moe_token_permute_gb300.workloads import make_inputs
    inp = make_inputs("mixtral", T, seed=4)
    wl = inp["wl"]
    hidden = inp["hidden"].cuda()
    ids = inp["topk_ids"].cuda()
    w = inp["topk_weights"].cuda()
    rows = inp["rows"].cuda()
    bufs = alloc_outputs(T, wl.K, wl.E, wl.H, torch.bfloat16)
    out = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")

    def step():
        mp.moe_permute(hidden, ids, bufs["offsets"], bufs["pidx"], bufs["inv"], bufs["ws"],
                       num_experts=wl.E, permuted_hidden_states=bufs["ph"])
        mp.moe_unpermute(rows, w, bufs["inv"], out)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [bufs[k].clone() for k in ("offsets", "pidx", "inv", "ph")] + [out.clone()]
    for k in ("offsets", "pidx", "inv"):
        bufs[k].fill_(-9)
    bufs["ph"].zero_()
    out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, [bufs[k] for k in ("offsets", "pidx", "inv", "ph")] + [out]):
        assert torch.equal(a, b)


def test_error_codes_through_binding():
    T, K, E = 64, 2, 8
    ids = torch.randint(0, E, (T, K), dtype=torch.int32, device="cuda")
    bufs = alloc_outputs(T, K, E, None, None)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    big_T = 100000
    big_ids = torch.zeros(big_T, K, dtype=torch.int32, device="cuda")
    with pytest.raises(mp.MoeError, match="workspace"):
        mp.moe_permute(None, big_ids, bufs["offsets"], torch.empty(big_T * K, dtype=torch.int32, device="cuda"),
                       torch.empty(big_T * K, dtype=torch.int32, device="cuda"), small, num_experts=E)
    with pytest.raises(mp.MoeError, match="invalid"):
        mp.moe_permute(None, ids, bufs["offsets"], bufs["pidx"], bufs["inv"], bufs["ws"],
                       num_experts=E, num_local_experts=4)
    assert mp.moe_permute_supported(torch.cuda.current_device())
