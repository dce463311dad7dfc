"""Seeded random configurations against the oracle.

Each case draws:
- a token count, often at the single-launch / routing-grid boundary;
- a top-k and an expert count, with or without an expert map (some with a
  bad map value);
- ids with duplicates and, sometimes, out-of-range values;
- a row width and dtype (fp8 rows with scales among them), and an id dtype.

The CUDA path must match the oracle bit for bit: the metadata, the gathered
rows and scales, the status flags and the unpermute output; and for bf16 rows
whose width is a multiple of 128, also the quantise-on-permute codes and
scales.
"""
import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
import oracle
from gpu_util import (assert_metadata_equal, assert_rows_equal_full, assert_unpermute_matches,
                      bits16, bytes_of, gpu_permute, gpu_unpermute, oracle_full)
from test_edges_gpu import custom_inputs
from test_quant_gpu import oracle_quant_permute, run_quant

pytestmark = pytest.mark.gpu

N_CASES = 48
MAX_ELEMS = 6_000_000  # cap on T*K*H (the unpermute input), so the oracle finishes quickly


def draw(seed):
    rng = np.random.default_rng(7919 + seed)
    K = int(rng.choice([1, 2, 3, 4, 6, 8, 8, 13, 32], p=[.1, .2, .1, .15, .1, .15, .05, .05, .1]))
    if rng.random() < 0.4:  # around the single launch's limits: 2048 rows (2 -> 4 rows per lane), 3072 (its end without a map)
        T = max(1, int(rng.choice([2048, 3072])) // K + int(rng.integers(-2, 3)))
    else:
        T = int(np.exp(rng.uniform(0, np.log(7000))))
    E = int(rng.integers(1, 300))
    emap, E_local = None, E
    if rng.random() < 0.35:
        E_local = int(rng.integers(1, min(E, 1024) + 1))
        emap = np.full(E, -1, dtype=np.int32)
        emap[rng.permutation(E)[:E_local]] = rng.permutation(E_local).astype(np.int32)
        if rng.random() < 0.25:
            emap[int(rng.integers(0, E))] = E_local + 3 if rng.random() < 0.5 else -4
        emap = torch.from_numpy(emap)
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    if rng.random() < 0.2:
        bad = rng.random((T, K)) < 0.01
        ids[bad] = rng.choice([-1, -7, E, E + 5], size=int(bad.sum()))
    kind = rng.choice(["bf16", "bf16", "fp16", "fp8", "fp32"])
    H = int(rng.choice([1, 8, 64, 100, 128, 256, 1024, 2048, 4096]))
    scale_cols = 0
    dtype = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8": torch.float8_e4m3fn,
             "fp32": torch.float32}[kind]
    if kind == "fp8":
        H = max(128, H // 128 * 128)
        scale_cols = H // 128
    if T * K * H > MAX_ELEMS:
        T = max(1, MAX_ELEMS // (K * H))
        ids = ids[:T]
    id_dtype = torch.int64 if rng.random() < 0.3 else torch.int32
    inp = custom_inputs(T, K, E, H, dtype=dtype, E_local=E_local, emap=emap,
                        ids=torch.from_numpy(np.ascontiguousarray(ids)), scale_cols=scale_cols,
                        seed=seed)
    return inp, id_dtype


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_config_matches_oracle(seed):
    inp, id_dtype = draw(seed)
    T, wl = inp["T"], inp["wl"]
    ref = oracle_full(inp)
    bufs = gpu_permute(inp, ids_dtype=id_dtype)
    assert_metadata_equal(bufs, ref)
    assert_rows_equal_full(inp, bufs, ref)
    assert mp.moe_read_status(bufs["ws"]) == ref["flags"]

    out = gpu_unpermute(inp["rows"], inp["topk_weights"],
                        torch.from_numpy(ref["inv_permuted_idx"]))
    ref_out, _ = oracle.unpermute(bits16(inp["rows"]), inp["topk_weights"].numpy(),
                                  ref["inv_permuted_idx"])
    assert_unpermute_matches(bits16(out), ref_out)

    if inp["hidden"].dtype == torch.bfloat16 and wl.H % 128 == 0:
        qref = oracle_quant_permute(inp["hidden"], inp)
        qbufs, codes, scales = run_quant(inp["hidden"], inp, ids_dtype=id_dtype)
        assert_metadata_equal(qbufs, qref)
        n = qref["n_valid"]
        np.testing.assert_array_equal(bytes_of(codes[:n]), qref["permuted_hidden"][:n])
        np.testing.assert_array_equal(scales[:n].cpu().numpy(), qref["permuted_scales"][:n])
        assert mp.moe_read_status(qbufs["ws"]) == qref["flags"]
