"""GPU parity of quantise-on-permute (moe_permute_quant_fp8) against the CPU
oracle: the oracle quantises every token row (per-token, per-128-column fp8
e4m3) and then permutes the codes and scales like any other rows.  Codes,
scales, offsets and both index maps must match bit for bit."""
import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
import oracle
from gpu_util import alloc_outputs, assert_bytes_equal, assert_metadata_equal, bits16, bytes_of
from test_edges_gpu import custom_inputs
from moe_token_permute_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

G = mp._binding.MOE_QUANT_GROUP


def bf16_rows(T, H, seed, device="cpu"):
    """bf16 N(0,1) rows with per-token magnitudes spread over ~2 decades, plus
    planted corner cases: an all-zero group, a tiny-valued group (e4m3
    subnormal codes) and a group with one large spike."""
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn(T, H, generator=g, device=device)
    x = x * torch.exp(torch.randn(T, 1, generator=g, device=device))
    if T > 0 and H >= 3 * G:
        x[0, 0:G] = 0.0
        x[0, G:2 * G] *= 1e-4
        x[T - 1, 2 * G:3 * G] *= 1e-3
        x[T - 1, 2 * G + 5] = 300.0
    return x.to(torch.bfloat16).contiguous()


def run_quant(hidden, inp, ids_dtype=torch.int32):
    wl = inp["wl"]
    T = hidden.shape[0]
    H = hidden.shape[1]
    bufs = alloc_outputs(T, wl.K, wl.e_local, E=wl.E)
    R = T * wl.K
    codes = torch.zeros(R, H, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(R, H // G, dtype=torch.float32, device="cuda")
    emap = None if inp["expert_map"] is None else inp["expert_map"].cuda()
    mp.moe_permute_quant_fp8(hidden.cuda(), inp["topk_ids"].to(device="cuda", dtype=ids_dtype),
                             bufs["offsets"], bufs["pidx"], bufs["inv"], bufs["ws"], codes, scales,
                             num_experts=wl.E, num_local_experts=wl.e_local, expert_map=emap)
    return bufs, codes, scales


def oracle_quant_permute(hidden, inp):
    wl = inp["wl"]
    q, s = oracle.quantize_fp8(bits16(hidden), G)
    return oracle.permute(inp["topk_ids"].cpu().numpy(), wl.E,
                          expert_map=None if inp["expert_map"] is None else inp["expert_map"].cpu().numpy(),
                          E_local=wl.e_local, hidden=q, scales=s)


# T*K <= 2048 takes the single-launch kernel, above it the routing grid plus
# the quantising gather: dsv3 T=256 / 257 (K=8) straddle the boundary.
CASES = [("dsv3", 1), ("dsv3", 128), ("dsv3", 256), ("dsv3", 257), ("dsv3", 4096),
         ("qwen3", 1024), ("mixtral", 512), ("dsv2lite", 256), ("dsv2lite", 8192), ("tiny", 16)]


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}-T{T}" for n, T in CASES])
def test_quant_permute_matches_oracle(name, T):
    inp = make_inputs(name, T, seed=5, with_rows=False)
    hidden = bf16_rows(T, WORKLOADS[name].H, seed=T + 7)
    ref = oracle_quant_permute(hidden, inp)
    bufs, codes, scales = run_quant(hidden, inp)
    assert_metadata_equal(bufs, ref)
    n = ref["n_valid"]
    np.testing.assert_array_equal(bytes_of(codes[:n]), ref["permuted_hidden"][:n])
    np.testing.assert_array_equal(scales[:n].cpu().numpy(), ref["permuted_scales"][:n])
    assert mp.moe_read_status(bufs["ws"]) == 0


@pytest.mark.parametrize("T", [200, 300])  # single launch, routing grid + gather
def test_quant_permute_int64_ids_and_one_group_rows(T):
    inp = make_inputs("qwen3", T, seed=6, with_rows=False)
    hidden = bf16_rows(T, G, seed=3)  # H = 128: a single group per row
    ref = oracle_quant_permute(hidden, inp)
    bufs, codes, scales = run_quant(hidden, inp, ids_dtype=torch.int64)
    assert_metadata_equal(bufs, ref)
    n = ref["n_valid"]
    np.testing.assert_array_equal(bytes_of(codes[:n]), ref["permuted_hidden"][:n])
    np.testing.assert_array_equal(scales[:n].cpu().numpy(), ref["permuted_scales"][:n])


def test_quant_permute_large_full():
    """The DeepSeek-V3-shaped layer at 32768 tokens (inputs drawn on the
    device): metadata, every kept row's codes and scales against the oracle
    (1.9 GB of codes)."""
    T = 32768
    inp = make_inputs("dsv3", T, seed=0, device="cuda", with_rows=False)
    hidden = bf16_rows(T, WORKLOADS["dsv3"].H, seed=1, device="cuda")
    bufs, codes, scales = run_quant(hidden, inp)
    ref = oracle_quant_permute(hidden, inp)
    assert_metadata_equal(bufs, ref)
    n = ref["n_valid"]
    assert_bytes_equal(bytes_of(codes[:n]), ref["permuted_hidden"][:n], "codes")
    np.testing.assert_array_equal(scales[:n].cpu().numpy().view(np.uint32),
                                  ref["permuted_scales"][:n].view(np.uint32))
    assert mp.moe_read_status(bufs["ws"]) == 0


@pytest.mark.parametrize("H,codes_off,scales_off", [
    (768, 0, 0),     # 6 groups a row: scales one by one, a half item at each row's end
    (2048, 0, 4),    # scales 4-byte aligned only: one by one
    (2048, 8, 0),    # codes 8-byte aligned only: the 8-byte code stores
    (1152, 8, 4),    # 9 groups, both narrow
])
def test_quant_permute_store_variants(H, codes_off, scales_off):
    """The quantising gather writes 16-byte code stores and float4 scale
    stores where the output rows allow it, and narrower ones otherwise; every
    variant must give the oracle's codes and scales bit for bit."""
    T = 600  # 4800 expanded rows: the routing grid and the quantising gather
    inp = make_inputs("qwen3", T, seed=H + codes_off, with_rows=False)
    wl = inp["wl"]
    hidden = bf16_rows(T, H, seed=H)
    ref = oracle_quant_permute(hidden, inp)
    R = T * wl.K
    bufs = alloc_outputs(T, wl.K, wl.e_local, E=wl.E)
    cflat = torch.zeros(R * H + codes_off, dtype=torch.uint8, device="cuda")
    sflat = torch.zeros(R * (H // G) + scales_off // 4, dtype=torch.float32, device="cuda")
    codes = cflat[codes_off:].view(R, H)
    scales = sflat[scales_off // 4:].view(R, H // G)
    mp.moe_permute_quant_fp8(hidden.cuda(), inp["topk_ids"].cuda(), bufs["offsets"], bufs["pidx"],
                             bufs["inv"], bufs["ws"], codes, scales, num_experts=wl.E)
    assert_metadata_equal(bufs, ref)
    n = ref["n_valid"]
    assert_bytes_equal(bytes_of(codes[:n]), ref["permuted_hidden"][:n], "codes")
    np.testing.assert_array_equal(scales[:n].cpu().numpy().view(np.uint32),
                                  ref["permuted_scales"][:n].view(np.uint32))


def test_quant_permute_rejects_bad_shapes():
    inp = make_inputs("tiny", 16, with_rows=False)
    wl = inp["wl"]
    bufs = alloc_outputs(16, wl.K, wl.E)
    ids = inp["topk_ids"].cuda()
    for H in (100, 64):  # not a whole number of 128-column groups
        h = torch.zeros(16, H, dtype=torch.bfloat16, device="cuda")
        c = torch.zeros(32, H, dtype=torch.uint8, device="cuda")
        s = torch.zeros(32, 1, dtype=torch.float32, device="cuda")
        with pytest.raises(mp.MoeError, match="invalid"):
            mp.moe_permute_quant_fp8(h, ids, bufs["offsets"], bufs["pidx"], bufs["inv"], bufs["ws"],
                                     c, s, num_experts=wl.E)
    flat = torch.zeros(16 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    h = flat[1:].view(16, 128)  # 2-byte aligned only
    c = torch.zeros(32, 128, dtype=torch.uint8, device="cuda")
    s = torch.zeros(32, 1, dtype=torch.float32, device="cuda")
    with pytest.raises(mp.MoeError, match="invalid"):
        mp.moe_permute_quant_fp8(h, ids, bufs["offsets"], bufs["pidx"], bufs["inv"], bufs["ws"],
                                 c, s, num_experts=wl.E)


def test_quant_permute_zero_tokens():
    inp = make_inputs("dsv3", 0, with_rows=False)
    wl = inp["wl"]
    bufs = alloc_outputs(0, wl.K, wl.E)
    h = torch.zeros(0, wl.H, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(0, wl.H, dtype=torch.uint8, device="cuda")
    s = torch.zeros(0, wl.H // G, dtype=torch.float32, device="cuda")
    mp.moe_permute_quant_fp8(h, inp["topk_ids"].cuda(), bufs["offsets"], bufs["pidx"], bufs["inv"],
                             bufs["ws"], c, s, num_experts=wl.E)
    assert bufs["offsets"].cpu().tolist() == [0] * (wl.E + 1)


def every_bf16_up_to(amax_bits):
    """Bit patterns of every finite bf16 value v with |v| <= the value of amax_bits."""
    mags = np.arange(0, 0x7F81, dtype=np.uint16)  # +0 .. +inf (exclusive of NaN)
    mags = mags[(mags <= amax_bits) & (mags < 0x7F80)]
    return np.concatenate([mags, mags | np.uint16(0x8000)])


# Group maxima (bf16 bits): 448 gives scale 1 (every e4m3 midpoint is hit exactly), powers of
# two, odd mantissas, the smallest subnormal and normal, and the largest finite bf16.
AMAX_BITS = [0x43E0, 0x3F80, 0x4040, 0x3F95, 0x4321, 0x0001, 0x0080, 0x0C00, 0x3000, 0x3C80,
             0x447F, 0x4B00, 0x5F00, 0x7F7F, 0x41C8, 0x3A83]


def test_quant_every_bf16_value_against_oracle():
    """Every finite bf16 value, under each group maximum above, quantised by the
    kernel (multiply by the reciprocal where it provably gives the IEEE
    quotient's code, the division elsewhere) against the oracle's division."""
    H = 1024
    groups = []
    for a in AMAX_BITS:
        vals = every_bf16_up_to(a)
        per = G - 1
        for i in range(0, len(vals), per):
            g = np.full(G, a, dtype=np.uint16)  # the maximum itself, then values <= it
            chunk = vals[i:i + per]
            g[1:1 + len(chunk)] = chunk
            groups.append(g)
    while len(groups) % (H // G):
        groups.append(np.zeros(G, dtype=np.uint16))
    bits = np.concatenate(groups).reshape(-1, H)
    T = bits.shape[0]
    hidden = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    inp = custom_inputs(T, 1, 1, H, ids=torch.zeros(T, 1, dtype=torch.int32), seed=0)
    ref = oracle_quant_permute(hidden, inp)
    bufs, codes, scales = run_quant(hidden, inp)
    np.testing.assert_array_equal(bytes_of(codes), ref["permuted_hidden"])
    np.testing.assert_array_equal(scales.cpu().numpy(), ref["permuted_scales"])
