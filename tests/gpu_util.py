"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import moe_token_permute_gb300 as mp
import oracle
import pins

DEV = "cuda"

# Unpermute tolerance stated for the path: |gpu - ref| <= 2^-7 |ref| + 1e-6,
# ref = the oracle's fp32 sum rounded to bf16.
UNPERMUTE_RTOL = 2.0 ** -7
UNPERMUTE_ATOL = 1e-6


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16/fp16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bytes_of(t: torch.Tensor) -> np.ndarray:
    """Any tensor -> its raw bytes [rows, row_bytes] on the host."""
    t = t.detach().cpu().contiguous()
    row_bytes = t.element_size() * int(np.prod(t.shape[1:], dtype=np.int64))
    return t.view(torch.uint8).numpy().reshape(t.shape[0], row_bytes)


def alloc_outputs(T, K, E_local, H=None, dtype=None, scale_cols=0, E=None, device=DEV):
    R = T * K
    out = dict(
        offsets=torch.full((E_local + 1,), -7, dtype=torch.int64, device=device),
        pidx=torch.full((R,), -7, dtype=torch.int32, device=device),
        inv=torch.full((R,), -7, dtype=torch.int32, device=device),
        ph=None, ps=None)
    if H is not None:
        out["ph"] = torch.zeros(R, H, dtype=dtype, device=device)
        if scale_cols:
            out["ps"] = torch.zeros(R, scale_cols, dtype=torch.float32, device=device)
    nbytes = mp.moe_permute_workspace_size(T, K, E if E is not None else E_local)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    mp.moe_permute_workspace_init(ws)
    out["ws"] = ws
    return out


def gpu_permute(inp, ids_dtype=torch.int32, metadata_only=False, bufs=None, device=DEV):
    """Run moe_permute on a make_inputs() dict; returns the device buffers."""
    wl = inp["wl"]
    T = inp["T"]
    hidden = inp["hidden"].to(device)
    scales = None if inp["scales"] is None else inp["scales"].to(device)
    ids = inp["topk_ids"].to(device=device, dtype=ids_dtype)
    emap = None if inp["expert_map"] is None else inp["expert_map"].to(device)
    if bufs is None:
        bufs = alloc_outputs(T, wl.K, wl.e_local, None if metadata_only else wl.H,
                             hidden.dtype, 0 if scales is None else scales.shape[1], E=wl.E,
                             device=device)
    mp.moe_permute(None if metadata_only else hidden, ids, bufs["offsets"], bufs["pidx"],
                   bufs["inv"], bufs["ws"], num_experts=wl.E, num_local_experts=wl.e_local,
                   expert_map=emap, hidden_scales=None if metadata_only else scales,
                   permuted_hidden_states=bufs["ph"], permuted_scales=bufs["ps"])
    return bufs


def oracle_route(inp):
    wl = inp["wl"]
    return oracle.permute(inp["topk_ids"].cpu().numpy(), wl.E,
                          expert_map=None if inp["expert_map"] is None
                          else inp["expert_map"].cpu().numpy(),
                          E_local=wl.e_local)


def assert_metadata_equal(bufs, ref):
    np.testing.assert_array_equal(bufs["offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(bufs["pidx"].cpu().numpy(), ref["permuted_idx"])
    np.testing.assert_array_equal(bufs["inv"].cpu().numpy(), ref["inv_permuted_idx"])


def assert_bytes_equal(got: np.ndarray, ref: np.ndarray, what: str, chunk_rows: int = 1 << 16):
    """Row-by-row byte equality of two [rows, row_bytes] arrays, compared in
    chunks so that gigabyte outputs need no gigabyte temporaries."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    for r0 in range(0, got.shape[0], chunk_rows):
        g, f = got[r0:r0 + chunk_rows], ref[r0:r0 + chunk_rows]
        if not np.array_equal(g, f):
            bad = np.flatnonzero((g != f).reshape(g.shape[0], -1).any(axis=1))
            raise AssertionError(f"{what}: {bad.size} rows differ from row {r0 + int(bad[0])} on")


def assert_rows_equal_full(inp, bufs, ref_full):
    """Every kept permuted row (p < N_valid) and scale row, bit for bit."""
    n = ref_full["n_valid"]
    assert_bytes_equal(bytes_of(bufs["ph"][:n]), ref_full["permuted_hidden"][:n],
                       "permuted_hidden_states")
    if bufs["ps"] is not None:
        assert_bytes_equal(bytes_of(bufs["ps"][:n]),
                           np.ascontiguousarray(ref_full["permuted_scales"][:n]).view(np.uint8),
                           "permuted_scales")


def oracle_full(inp):
    """Oracle permute including the row copy (rows handed over as raw bytes)."""
    wl = inp["wl"]
    hidden = bytes_of(inp["hidden"])
    return oracle.permute(inp["topk_ids"].cpu().numpy(), wl.E,
                          expert_map=None if inp["expert_map"] is None
                          else inp["expert_map"].cpu().numpy(),
                          E_local=wl.e_local, hidden=hidden,
                          scales=None if inp["scales"] is None else inp["scales"].cpu().numpy())


def gpu_unpermute(rows, weights, inv, ws=None, device=DEV):
    T, K = weights.shape
    out = torch.full((T, rows.shape[1]), float("nan"), dtype=torch.bfloat16, device=device)
    mp.moe_unpermute(rows.to(device), weights.to(device), inv.to(device), out, workspace=ws)
    return out


def assert_unpermute_matches(got_bits: np.ndarray, ref_bits: np.ndarray):
    """Every element within 2^-7*|ref| + 1e-6 of the oracle, and in fact equal
    bit for bit: both sides take the same fp32 operations in the same order.
    Elements equal in their bits pass both; the tolerance is evaluated on the
    others, so that the check stays cheap on gigabyte outputs."""
    assert got_bits.shape == ref_bits.shape
    diff = got_bits != ref_bits
    mism = int(np.count_nonzero(diff))
    if mism == 0:
        return
    got = pins.bf16_bits_to_f64(got_bits[diff])
    ref = pins.bf16_bits_to_f64(ref_bits[diff])
    err = np.abs(got - ref)
    bound = UNPERMUTE_RTOL * np.abs(ref) + UNPERMUTE_ATOL
    assert np.all(err <= bound), f"max excess {float((err - bound).max())}"
    raise AssertionError(f"{mism} elements differ in their bits (within tolerance)")
