"""One workspace across many routing calls.

The routing grid's blocks exchange their per-expert histograms through a
table in the workspace whose entries carry a per-call tag; a later call must
never take an entry an earlier call left for one of its own.  These tests
reuse one workspace across shapes whose table extent grows and shrinks
(different block counts and expert counts), and across more calls than there
are distinct tags, and compare every call's metadata with the oracle.
"""
import pytest
import torch

import moe_token_permute_gb300 as mp
from gpu_util import alloc_outputs, assert_metadata_equal, gpu_permute, oracle_route, oracle_full, \
    assert_rows_equal_full
from moe_token_permute_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


def shared_workspace(shapes):
    nbytes = max(mp.moe_permute_workspace_size(T, K, E) for T, K, E in shapes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)  # whatever the allocation held; init must clear it all
    mp.moe_permute_workspace_init(ws)
    return ws


# (workload, T, with rows): table extents 128x128, 8x8, 64x256, 79x256 (a large table:
# rounds of 8 rows per lane), 18x16, 128x128, 59x8, 1x8
SEQUENCE = [("qwen3", 16384, False), ("mixtral", 4096, True), ("dsv3", 8192, False),
            ("dsv3", 20000, False), ("dsv2lite", 3000, True), ("qwen3", 16384, False),
            ("mixtral", 30000, False), ("mixtral", 1024, True), ("qwen3", 5000, True)]


def test_shapes_growing_and_shrinking_share_one_workspace():
    inps = [make_inputs(name, T, seed=10 + i, with_rows=rows)
            for i, (name, T, rows) in enumerate(SEQUENCE)]
    ws = shared_workspace([(inp["T"], inp["wl"].K, inp["wl"].E) for inp in inps])
    for inp, (name, T, rows) in zip(inps, SEQUENCE):
        wl = inp["wl"]
        bufs = alloc_outputs(T, wl.K, wl.e_local, wl.H if rows else None,
                             inp["hidden"].dtype if rows else None,
                             0 if (not rows or inp["scales"] is None) else inp["scales"].shape[1],
                             E=wl.E)
        bufs["ws"] = ws
        gpu_permute(inp, metadata_only=not rows, bufs=bufs)
        if rows:
            ref = oracle_full(inp)
            assert_metadata_equal(bufs, ref)
            assert_rows_equal_full(inp, bufs, ref)
        else:
            assert_metadata_equal(bufs, oracle_route(inp))
    assert mp.moe_read_status(ws) == 0


def test_more_calls_than_tags():
    """300 back-to-back calls alternating two shapes (table extents 32x128 and
    16x8) on one workspace; every call's metadata is checked on the device."""
    a = make_inputs("qwen3", 4096, seed=21, with_rows=False)
    b = make_inputs("mixtral", 8192, seed=22, with_rows=False)
    ws = shared_workspace([(x["T"], x["wl"].K, x["wl"].E) for x in (a, b)])
    cases = []
    for inp in (a, b):
        wl = inp["wl"]
        ref = oracle_route(inp)
        bufs = alloc_outputs(inp["T"], wl.K, wl.e_local, E=wl.E)
        bufs["ws"] = ws
        expect = {k: torch.from_numpy(ref[v]).cuda() for k, v in
                  (("offsets", "offsets"), ("pidx", "permuted_idx"), ("inv", "inv_permuted_idx"))}
        cases.append((inp, bufs, expect))
    bad = []
    for i in range(300):
        inp, bufs, expect = cases[i % 2]
        for k in expect:
            bufs[k].fill_(-5)
        gpu_permute(inp, metadata_only=True, bufs=bufs)
        if not all(torch.equal(bufs[k], expect[k]) for k in expect):
            bad.append(i)
    assert bad == []
    assert mp.moe_read_status(ws) == 0


def test_graph_replays_alternating_on_one_workspace():
    """Two CUDA graphs (different shapes, so different table extents) captured
    on one workspace and replayed alternately 150 times: each replay takes its
    table tag from the workspace, not from the captured arguments, so every
    replay's metadata must match the oracle."""
    a = make_inputs("qwen3", 3000, seed=31, with_rows=False)
    b = make_inputs("dsv3", 6000, seed=32, with_rows=False)
    ws = shared_workspace([(x["T"], x["wl"].K, x["wl"].E) for x in (a, b)])
    cases = []
    for inp in (a, b):
        wl = inp["wl"]
        ref = oracle_route(inp)
        bufs = alloc_outputs(inp["T"], wl.K, wl.e_local, E=wl.E)
        bufs["ws"] = ws
        ids = inp["topk_ids"].cuda()
        expect = {k: torch.from_numpy(ref[v]).cuda() for k, v in
                  (("offsets", "offsets"), ("pidx", "permuted_idx"), ("inv", "inv_permuted_idx"))}

        def call(ids=ids, bufs=bufs, wl=wl):
            mp.moe_permute(None, ids, bufs["offsets"], bufs["pidx"], bufs["inv"], bufs["ws"],
                           num_experts=wl.E, num_local_experts=wl.e_local)

        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            call()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        # the graph reads ids by address: keep the tensor (and the closure) alive
        cases.append((g, bufs, expect, ids, call))
    bad = []
    for i in range(150):
        g, bufs, expect, _, _ = cases[i % 2]
        for k in expect:
            bufs[k].fill_(-5)
        g.replay()
        torch.cuda.synchronize()
        if not all(torch.equal(bufs[k], expect[k]) for k in expect):
            bad.append(i)
    assert bad == []
    assert mp.moe_read_status(ws) == 0
