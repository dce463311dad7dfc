"""Permute with an expert map above 4096 expanded rows, against the oracle.

With an expert map and 16-byte aligned rows, moe_permute routes each block of
tokens and copies the rows of the tokens that keep one in a single launch.
Each case below is shaped to drive one of that kernel's paths, and each is
compared with the CPU oracle element by element (offsets, both index maps,
every kept row and scale row, the status flags):

- 2 or 4 rows per lane (up to 1024 or 2048 expanded rows per block);
- rows split into several chunks, the last one shorter;
- stage refills: more row chunks per block than ring stages, over many rounds;
- fp8 rows with their scale rows;
- a large local expert count (the ranking arrays leave room for few stages);
- a map so sparse that some blocks keep no token at all;
- ids and map values out of range (dropped and flagged), int64 ids.
"""
import numpy as np
import pytest
import torch

from test_edges_gpu import check_case, custom_inputs

pytestmark = pytest.mark.gpu


def expert_map(E, E_local, seed, bad=None):
    """E_local of E experts local (ids 0..E_local-1 in a random order), the rest -1;
    `bad` plants one out-of-range value."""
    rng = np.random.default_rng(seed)
    m = np.full(E, -1, dtype=np.int32)
    m[rng.permutation(E)[:E_local]] = rng.permutation(E_local).astype(np.int32)
    if bad is not None:
        m[int(rng.integers(0, E))] = bad
    return torch.from_numpy(m)


# name: (T, K, E, E_local, H, dtype, scale_cols)
CASES = {
    "one_row_per_token_4_per_lane": (200000, 1, 64, 16, 16, torch.bfloat16, 0),
    "top8_4_rows_per_lane": (30000, 8, 128, 32, 256, torch.bfloat16, 0),
    "wide_rows_ragged_chunks": (3000, 2, 16, 5, 5000, torch.bfloat16, 0),
    "fp8_rows_with_scales": (2000, 8, 256, 64, 7168, torch.float8_e4m3fn, 56),
    "1024_local_experts": (1100, 4, 2048, 1024, 64, torch.bfloat16, 0),
    "one_local_expert": (5000, 2, 64, 1, 128, torch.bfloat16, 0),
    "many_refill_rounds": (20000, 1, 2048, 1024, 4096, torch.bfloat16, 0),
    "fp32_rows": (3000, 3, 40, 10, 24, torch.float32, 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_expert_map_permute_matches_oracle(name):
    T, K, E, E_local, H, dtype, scale_cols = CASES[name]
    emap = expert_map(E, E_local, seed=T + K)
    inp = custom_inputs(T, K, E, H, dtype=dtype, E_local=E_local, emap=emap,
                        scale_cols=scale_cols, seed=T)
    ref, _ = check_case(inp, unpermute=False)
    if name == "one_local_expert":
        # about 3% of the tokens keep a row: most blocks keep a few, some none
        assert 0 < ref["n_valid"] < T * K // 10


@pytest.mark.parametrize("id_dtype", [torch.int32, torch.int64])
def test_expert_map_out_of_range_ids_and_map_values(id_dtype):
    T, K, E, E_local, H = 4000, 3, 32, 8, 96
    emap = expert_map(E, E_local, seed=5, bad=E_local + 2)
    g = torch.Generator().manual_seed(6)
    ids = torch.randint(0, E, (T, K), generator=g, dtype=torch.int32)
    ids[::97, 1] = E + 3   # id past the last expert
    ids[5::131, 2] = -2    # negative id
    inp = custom_inputs(T, K, E, H, E_local=E_local, emap=emap, ids=ids, seed=7)
    check_case(inp, expect_flags=1 | 2, unpermute=False, ids_dtype=id_dtype)
