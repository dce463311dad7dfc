"""Two serving streams at once, each with its own workspace.

A serving process may run several micro-batches on separate CUDA streams.
Each stream here owns a workspace and output buffers and issues permute +
unpermute calls back to back, with no synchronisation between the streams,
so the calls of both overlap on the GPU.  The batches are sized to take the
cooperative kernels (the routing grid with its gather; the single-launch
expert-map kernel), whose blocks wait on one another through their own
workspace's table: calls on different workspaces must not interfere.  After
the calls every output is compared with the CPU oracle element by element and
both status words must be clear.
"""
import numpy as np
import pytest
import torch

import moe_token_permute_gb300 as mp
from gpu_util import (alloc_outputs, assert_metadata_equal, assert_rows_equal_full,
                      assert_unpermute_matches, bits16, oracle_full)
from moe_token_permute_gb300.workloads import make_inputs
import oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


class Lane:
    """One stream's inputs, buffers and workspace."""

    def __init__(self, name, T, seed):
        self.inp = make_inputs(name, T, seed=seed, with_rows=True)
        wl = self.inp["wl"]
        sc = self.inp["scales"]
        self.bufs = alloc_outputs(T, wl.K, wl.e_local, wl.H, self.inp["hidden"].dtype,
                                  0 if sc is None else sc.shape[1], E=wl.E, device=DEV)
        self.hidden = self.inp["hidden"].to(DEV)
        self.scales = None if sc is None else sc.to(DEV)
        self.ids = self.inp["topk_ids"].to(DEV)
        self.emap = None if self.inp["expert_map"] is None else self.inp["expert_map"].to(DEV)
        self.rows = self.inp["rows"].to(DEV)
        self.w = self.inp["topk_weights"].to(DEV)
        self.out = torch.empty(T, wl.H, dtype=torch.bfloat16, device=DEV)
        self.stream = torch.cuda.Stream()

    def call(self):
        wl, b = self.inp["wl"], self.bufs
        mp.moe_permute(self.hidden, self.ids, b["offsets"], b["pidx"], b["inv"], b["ws"],
                       num_experts=wl.E, num_local_experts=wl.e_local, expert_map=self.emap,
                       hidden_scales=self.scales, permuted_hidden_states=b["ph"],
                       permuted_scales=b["ps"], stream=self.stream)
        mp.moe_unpermute(self.rows, self.w, b["inv"], self.out, workspace=b["ws"],
                         stream=self.stream)


@pytest.mark.parametrize("pair", [(("mixtral", 4096), ("dsv2lite", 8192)),
                                  (("qwen3", 8192), ("mixtral", 4096))],
                         ids=["route-grid+expert-map", "route-grid+route-grid"])
def test_two_streams_overlap(pair):
    lanes = [Lane(name, T, seed=31 + i) for i, (name, T) in enumerate(pair)]
    torch.cuda.synchronize()
    for _ in range(20):
        for lane in lanes:
            lane.call()
    torch.cuda.synchronize()
    for lane in lanes:
        assert mp.moe_read_status(lane.bufs["ws"]) == 0
        ref = oracle_full(lane.inp)
        assert_metadata_equal(lane.bufs, ref)
        assert_rows_equal_full(lane.inp, lane.bufs, ref)
        want, _ = oracle.unpermute(bits16(lane.inp["rows"]), lane.inp["topk_weights"].numpy(),
                                   lane.bufs["inv"].cpu().numpy())
        assert_unpermute_matches(bits16(lane.out), want)
