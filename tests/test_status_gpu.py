"""moe_permute_read_status, the asynchronous read of the workspace status
word: captured into a CUDA graph together with the permute it follows, it
copies the flags into device memory or pinned host memory on every replay,
with no host synchronisation inside the graph; with clear_after_read the word
starts the next step at zero.  The flags it reports are compared with the
oracle's on the same inputs."""
import ctypes

import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
import oracle
from moe_token_permute_gb300 import _binding as b

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [300, 3000])  # single-launch kernel; routing grid + gather
def test_async_status_read_inside_a_cuda_graph(T):
    K, E, H = 4, 16, 64
    g = torch.Generator().manual_seed(T)
    ids = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32)
    bad = ids.clone()
    bad[T // 3, 1] = 99   # outside [0, E): dropped and flagged
    bad[T - 1, 0] = -5
    ref_bad = oracle.permute(bad.numpy(), E)
    ref_good = oracle.permute(ids.numpy(), E)
    assert ref_bad["flags"] == mp.MOE_FLAG_ID_OUT_OF_RANGE and ref_good["flags"] == 0

    dev = "cuda"
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16).to(dev)
    d_ids = bad.to(dev)
    off = torch.empty(E + 1, dtype=torch.int64, device=dev)
    pidx = torch.empty(T * K, dtype=torch.int32, device=dev)
    inv = torch.empty(T * K, dtype=torch.int32, device=dev)
    ph = torch.empty(T * K, H, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mp.moe_permute_workspace_size(T, K, E), dtype=torch.uint8, device=dev)
    mp.moe_permute_workspace_init(ws)
    seen_dev = torch.full((1,), -1, dtype=torch.int32, device=dev)
    seen_host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    after_clear = torch.full((1,), -1, dtype=torch.int32, device=dev)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            mp.moe_permute(hidden, d_ids, off, pidx, inv, ws, num_experts=E,
                           permuted_hidden_states=ph, stream=s)
            mp.moe_permute_read_status(ws, seen_dev, stream=s)
            mp.moe_permute_read_status(ws, seen_host, clear_after_read=True, stream=s)
            mp.moe_permute_read_status(ws, after_clear, stream=s)
    torch.cuda.synchronize()
    for step_ids, ref in ((bad, ref_bad), (ids, ref_good), (bad, ref_bad)):
        d_ids.copy_(step_ids.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        assert int(seen_dev.item()) == ref["flags"]
        assert int(seen_host[0]) == ref["flags"]
        assert int(after_clear.item()) == 0
        np.testing.assert_array_equal(off.cpu().numpy(), ref["offsets"])
        np.testing.assert_array_equal(inv.cpu().numpy(), ref["inv_permuted_idx"])
    assert mp.moe_read_status(ws) == 0


def test_async_status_read_refuses_pageable_host_memory():
    ws = torch.empty(mp.moe_permute_workspace_size(16, 2, 8), dtype=torch.uint8, device="cuda")
    mp.moe_permute_workspace_init(ws)
    pageable = (ctypes.c_uint32 * 4)()
    rc = b.lib().moe_permute_read_status(ws.data_ptr(), ctypes.addressof(pageable), 0,
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == b.MOE_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        mp.moe_permute_read_status(ws, torch.zeros(1, dtype=torch.int32))  # not pinned
    torch.cuda.synchronize()
