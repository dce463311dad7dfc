"""The hand-worked cases of tests/golden/hand_worked.json through the CUDA path.

Every other GPU test compares the kernels with the CPU oracle; this one holds
them to the values worked out by hand from the definitions, with no program in
between: the routing metadata of the permute ("permute/unpermute kernel for moe
optimization" (vLLM PR #14568), description: expand each token to its K rows,
order them by expert, stable by row), the fp32 k-ordered unpermute sum rounded
once to bf16, the batched layout, and the per-128-column fp8 quantisation
("[Kernels] MoE refactor" (vLLM PR #19636), bot summary).  The status word is
compared with each case's flags.
"""
import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
from pins import f64_to_bf16_bits_exact, load_golden

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
G = load_golden()


def workspace(T, K, E):
    ws = torch.empty(mp.moe_permute_workspace_size(max(T, 1), K, E), dtype=torch.uint8, device=DEV)
    mp.moe_permute_workspace_init(ws)
    return ws


def bf16_rows(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).to(DEV).view(torch.bfloat16)


@pytest.mark.parametrize("case", G["routing"], ids=lambda c: c["name"])
def test_golden_routing(case):
    ids = torch.tensor(case["topk_ids"], dtype=torch.int32, device=DEV)
    T, K = ids.shape
    E, E_local = case["E"], case["E_local"]
    emap = (torch.tensor(case["expert_map"], dtype=torch.int32, device=DEV)
            if case["expert_map"] is not None else None)
    # row t holds the value t + 1 in every column, so each permuted row names its token
    H = 64
    hidden = (torch.arange(T, device=DEV, dtype=torch.float32) + 1).repeat_interleave(H).view(T, H)
    hidden = hidden.to(torch.bfloat16)
    R = T * K
    off = torch.full((E_local + 1,), -7, dtype=torch.int64, device=DEV)
    pidx = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    ph = torch.zeros(R, H, dtype=torch.bfloat16, device=DEV)
    ws = workspace(T, K, E)
    mp.moe_permute(hidden, ids, off, pidx, inv, ws, num_experts=E, num_local_experts=E_local,
                   expert_map=emap, permuted_hidden_states=ph)
    assert mp.moe_read_status(ws) == case["flags"]
    assert off.tolist() == case["offsets"]
    assert pidx.tolist() == case["permuted_idx"]
    assert inv.tolist() == case["inv_permuted_idx"]
    n_valid = case["offsets"][-1]
    want = torch.tensor([r // K + 1 for r in case["permuted_idx"][:n_valid]],
                        dtype=torch.float32, device=DEV)
    assert torch.equal(ph[:n_valid].float(), want[:, None].expand(n_valid, H))


@pytest.mark.parametrize("case", G["unpermute"], ids=lambda c: c["name"])
def test_golden_unpermute(case):
    rows = bf16_rows(f64_to_bf16_bits_exact(case["rows"]))
    if "topk_weights_f32_bits" in case:
        w = np.array(case["topk_weights_f32_bits"], np.uint32).view(np.float32)
    else:
        w = np.array(case["topk_weights"], np.float32)
    w = torch.from_numpy(w).to(DEV)
    inv = torch.tensor(case["inv_permuted_idx"], dtype=torch.int32, device=DEV)
    T, K = w.shape
    out = torch.full((T, rows.shape[1]), 123.0, dtype=torch.bfloat16, device=DEV)
    ws = workspace(T, K, 4)
    mp.moe_unpermute(rows, w, inv, out, workspace=ws)
    assert mp.moe_read_status(ws) == case.get("flags", 0)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16).tolist()
    assert got == case["out_bf16_bits"]


@pytest.mark.parametrize("case", G["batched"], ids=lambda c: c["name"])
def test_golden_batched(case):
    ids = torch.tensor(case["topk_ids"], dtype=torch.int32, device=DEV)
    T, K = ids.shape
    E, E_local, M = case["E"], case["E_local"], case["M"]
    emap = (torch.tensor(case["expert_map"], dtype=torch.int32, device=DEV)
            if case["expert_map"] is not None else None)
    counts = torch.full((E_local,), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((T * K,), -7, dtype=torch.int32, device=DEV)
    ws = workspace(T, K, E)
    mp.moe_permute_batched(None, ids, counts, inv, ws, num_experts=E, num_local_experts=E_local,
                           max_rows_per_expert=M, expert_map=emap)
    assert mp.moe_read_status(ws) == case["flags"]
    assert counts.tolist() == case["expert_num_tokens"]
    assert inv.tolist() == case["inv_permuted_idx"]


def test_golden_quantize_fp8():
    q = G["quantize_fp8"]
    group, groups = q["group"], q["groups"]
    H = group * len(groups)
    x = np.zeros((1, H), np.float32)
    for gi, grp in enumerate(groups):
        for i, v in grp["nonzero"].items():
            x[0, gi * group + int(i)] = v
    hidden = bf16_rows(f64_to_bf16_bits_exact(x))
    ids = torch.zeros(1, 1, dtype=torch.int32, device=DEV)
    off = torch.empty(2, dtype=torch.int64, device=DEV)
    pidx = torch.empty(1, dtype=torch.int32, device=DEV)
    inv = torch.empty(1, dtype=torch.int32, device=DEV)
    codes = torch.empty(1, H, dtype=torch.uint8, device=DEV)
    scales = torch.empty(1, H // group, dtype=torch.float32, device=DEV)
    ws = workspace(1, 1, 1)
    mp.moe_permute_quant_fp8(hidden, ids, off, pidx, inv, ws, codes, scales, num_experts=1)
    assert mp.moe_read_status(ws) == 0
    got_codes = codes.cpu().numpy()[0]
    got_scales = scales.cpu().numpy()[0]
    for gi, grp in enumerate(groups):
        want = np.zeros(group, np.uint8)
        for i, c in grp["codes_nonzero"].items():
            want[int(i)] = c
        assert got_codes[gi * group:(gi + 1) * group].tolist() == want.tolist(), grp["name"]
        if grp["scale_is"] == "1":
            assert got_scales[gi] == np.float32(1.0), grp["name"]
        else:
            num = float(grp["scale_is"].split("fp32(")[1].split(")")[0])
            assert got_scales[gi] == np.float32(num) / np.float32(448.0), grp["name"]
