"""The seeded input recipe (moe_token_permute_gb300/workloads.py) against the
workload table it is meant to follow: the layer shapes, dtypes and routing
of the Mixtral, Qwen3-30B-A3B, DeepSeek-V2-Lite and DeepSeek-V3 MoE layers
and the tiny case.  Every parity test and the benchmark draw from here."""
import numpy as np
import pytest
import torch

from moe_token_permute_gb300.workloads import FP8_BLOCK, FP8_MAX, WORKLOADS, make_inputs

SHAPES = {  # name: (H, E, E_local, K, hidden dtype, T sweep)
    "tiny": (128, 8, 8, 2, torch.bfloat16, (16,)),
    "mixtral": (4096, 8, 8, 2, torch.bfloat16, (1, 32, 512, 4096, 16384)),
    "qwen3": (2048, 128, 128, 8, torch.bfloat16, (1, 64, 1024, 8192, 16384)),
    "dsv2lite": (2048, 64, 16, 6, torch.bfloat16, (1, 256, 8192)),
    "dsv3": (7168, 256, 256, 8, torch.float8_e4m3fn, (1, 128, 4096, 32768)),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_shapes_and_dtypes(name):
    H, E, EL, K, dt, sweep = SHAPES[name]
    wl = WORKLOADS[name]
    assert (wl.H, wl.E, wl.e_local, wl.K, wl.T_sweep) == (H, E, EL, K, sweep)
    T = 24
    inp = make_inputs(name, T, seed=3)
    assert inp["hidden"].shape == (T, H) and inp["hidden"].dtype == dt
    assert inp["topk_ids"].shape == (T, K) and inp["topk_ids"].dtype == torch.int32
    assert inp["topk_weights"].shape == (T, K) and inp["topk_weights"].dtype == torch.float32
    assert inp["rows"].shape == (T * K, H) and inp["rows"].dtype == torch.bfloat16
    if dt == torch.float8_e4m3fn:
        assert inp["scales"].shape == (T, H // FP8_BLOCK) and inp["scales"].dtype == torch.float32
    else:
        assert inp["scales"] is None
    if EL == E:
        assert inp["expert_map"] is None
    else:
        assert inp["expert_map"].shape == (E,) and inp["expert_map"].dtype == torch.int32


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_k_distinct_experts_per_token_in_range(name):
    inp = make_inputs(name, 300, seed=5, with_rows=False)
    ids = inp["topk_ids"].numpy()
    E, K = inp["wl"].E, inp["wl"].K
    assert ids.min() >= 0 and ids.max() < E
    assert all(len(set(row)) == K for row in ids.tolist())


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_weights_are_a_softmax(name):
    w = make_inputs(name, 200, seed=6, with_rows=False)["topk_weights"].double()
    assert bool((w > 0).all())
    np.testing.assert_allclose(w.sum(dim=1).numpy(), 1.0, atol=1e-6)


def test_expert_map_marks_16_local_experts_in_global_order():
    m = make_inputs("dsv2lite", 4, seed=7, with_rows=False)["expert_map"].numpy()
    local = np.nonzero(m >= 0)[0]
    assert len(local) == 16 and (m[m < 0] == -1).all()
    # local ids 0..15 ascend with the global id
    np.testing.assert_array_equal(m[local], np.arange(16))
    # a different seed picks a different set
    m2 = make_inputs("dsv2lite", 4, seed=8, with_rows=False)["expert_map"].numpy()
    assert not np.array_equal(m, m2)


def test_uniform_routing_is_balanced():
    ids = make_inputs("mixtral", 16384, seed=9, with_rows=False)["topk_ids"].numpy()
    counts = np.bincount(ids.ravel(), minlength=8)
    expect = 16384 * 2 / 8
    assert np.abs(counts - expect).max() < 0.03 * expect


@pytest.mark.parametrize("name,s", [("qwen3", 1.2), ("dsv3", 1.0)])
def test_zipf_routing_is_skewed(name, s):
    wl = WORKLOADS[name]
    assert wl.routing == "zipf" and wl.zipf_s == s
    ids = make_inputs(name, 4096, seed=10, with_rows=False)["topk_ids"].numpy()
    counts = np.sort(np.bincount(ids.ravel(), minlength=wl.E))[::-1]
    # the most popular expert takes far more than a uniform share; the tail far less
    uniform = 4096 * wl.K / wl.E
    assert counts[0] > 8 * uniform
    assert counts[wl.E // 2] < uniform
    # and at the small sweep points some experts receive no row at all
    small = make_inputs(name, wl.T_sweep[1], seed=0, with_rows=False)["topk_ids"].numpy()
    assert len(np.unique(small)) < wl.E


def test_fp8_activations_use_the_block_maximum():
    inp = make_inputs("dsv3", 16, seed=11, with_rows=False)
    codes = inp["hidden"].float().reshape(16, -1, FP8_BLOCK)
    # scale = block amax / 448, so every block's largest code is exactly +-448
    np.testing.assert_array_equal(codes.abs().amax(dim=-1).numpy(), FP8_MAX)
    assert bool((inp["scales"] > 0).all())
    # codes * scale recovers N(0,1)-sized values
    x = codes * inp["scales"].unsqueeze(-1)
    assert 0.8 < float(x.std()) < 1.2


def test_seeded_and_rows_drawn_last():
    a = make_inputs("qwen3", 50, seed=12)
    b = make_inputs("qwen3", 50, seed=12, with_rows=False)
    c = make_inputs("qwen3", 50, seed=13, with_rows=False)
    for k in ("hidden", "topk_ids", "topk_weights"):
        assert torch.equal(a[k], b[k])
    assert b["rows"] is None
    assert not torch.equal(a["topk_ids"], c["topk_ids"])
