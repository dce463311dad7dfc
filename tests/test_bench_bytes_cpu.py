"""The benchmark's algorithmic byte counts, checked against the bytes of the
arrays each call must read and write, counted on small routed examples, and
against the figures the headline workload reports."""
import numpy as np
import pytest
import torch

import bench


def brute_counts(ids, emap, E):
    """(tokens with a kept row, kept rows) by plain loops."""
    kept_tokens, kept_rows = 0, 0
    for row in ids:
        k = 0
        for g in row:
            ok = 0 <= g < E and (emap is None or emap[g] >= 0)
            k += ok
        kept_tokens += k > 0
        kept_rows += k
    return kept_tokens, kept_rows


@pytest.mark.parametrize("with_map", [False, True])
def test_routing_counts(with_map):
    rng = np.random.default_rng(5)
    T, K, E = 37, 3, 9
    ids = rng.integers(-1, E + 1, size=(T, K)).astype(np.int32)
    emap = np.array([0, -1, 1, -1, 2, 3, -1, 4, -1], dtype=np.int32) if with_map else None
    got = bench.routing_counts(torch.from_numpy(ids), None if emap is None else
                               torch.from_numpy(emap), E, K)
    assert got == brute_counts(ids.tolist(), None if emap is None else emap.tolist(), E)


def test_permute_and_unpermute_bytes_match_array_sizes():
    T, K, H, E_L, elem, sc = 7, 3, 40, 5, 2, 0
    Tv, Nv = 6, 15
    R = T * K
    ids = np.zeros((T, K), np.int32).nbytes
    src_rows = Tv * H * elem               # each kept token's row read once
    dst_rows = Nv * H * elem               # one write per kept row
    maps = np.zeros(R, np.int32).nbytes * 2  # permuted_idx + inv_permuted_idx
    offsets = np.zeros(E_L + 1, np.int64).nbytes
    assert bench.permute_bytes(T, H, K, E_L, elem, sc, Tv, Nv) == \
        ids + src_rows + dst_rows + maps + offsets
    weights = np.zeros((T, K), np.float32).nbytes
    inv = np.zeros(R, np.int32).nbytes
    out = np.zeros((T, H), np.uint16).nbytes
    assert bench.unpermute_bytes(T, H, K, Nv) == inv + weights + Nv * H * 2 + out
    assert bench.metadata_bytes(T, K, E_L) == ids + maps + offsets


def test_fp8_and_quant_bytes():
    T, K, H, E_L, Tv, Nv = 4, 2, 256, 3, 4, 7
    sc = H // 128
    row = H * 1 + sc * 4                    # fp8 codes plus fp32 scales
    assert bench.permute_bytes(T, H, K, E_L, 1, sc, Tv, Nv) == \
        T * K * 4 + Tv * row + Nv * row + 2 * T * K * 4 + (E_L + 1) * 8
    # quantise-on-permute reads bf16 rows, writes fp8 codes and scales
    assert bench.quant_permute_bytes(T, H, K, E_L, Tv, Nv) == \
        T * K * 4 + Tv * H * 2 + Nv * (H + sc * 4) + 2 * T * K * 4 + (E_L + 1) * 8


def test_headline_workload_bytes():
    """Mixtral-shaped layer, T = 16384, uniform distinct top-2: every row is
    kept, so T_v = T and N_v = 2T; the step moves 806 MB."""
    T, H, K, E = 16384, 4096, 2, 8
    assert bench.permute_bytes(T, H, K, E, 2, 0, T, 2 * T) == 403_046_472
    assert bench.unpermute_bytes(T, H, K, 2 * T) == 402_915_328
