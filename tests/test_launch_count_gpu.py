"""How many kernels one call launches, read from a CUDA graph of that call.

bench.py reports `gpu_launches` from Setup.launches_per_permute (and one per
moe_unpermute).  Here one call is captured into a CUDA graph and its kernel
nodes are counted through the driver (cuGraphGetNodes / cuGraphNodeGetType),
at batch sizes on both sides of every dispatch boundary: the single-launch
kernel (up to 2048, 3072 or 4096 expanded rows depending on the call), the
single-launch expert-map kernel, and the routing grid plus a gather.
"""
import ctypes

import pytest
import torch

import bench

pytestmark = pytest.mark.gpu

CU_GRAPH_NODE_TYPE_KERNEL = 0


def kernel_nodes(fn):
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this torch keeps no raw CUDA graph")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.synchronize()
    raw = ctypes.c_void_p(int(g.raw_cuda_graph()))
    cu = ctypes.CDLL("libcuda.so.1")
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(raw, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * max(1, n.value))()
    assert cu.cuGraphGetNodes(raw, nodes, ctypes.byref(n)) == 0
    kinds = []
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kinds.append(t.value)
    del g
    return sum(1 for k in kinds if k == CU_GRAPH_NODE_TYPE_KERNEL), len(kinds)


# (workload, T): expanded rows T*K on both sides of each boundary
CASES = [("mixtral", 1), ("mixtral", 1024), ("mixtral", 1536), ("mixtral", 1537), ("mixtral", 4096),
         ("qwen3", 64), ("qwen3", 384), ("qwen3", 385),
         ("dsv2lite", 256), ("dsv2lite", 682), ("dsv2lite", 683), ("dsv2lite", 8192),
         ("dsv3", 256), ("dsv3", 257), ("dsv3", 384), ("dsv3", 385)]


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}-T{t}" for n, t in CASES])
def test_permute_and_unpermute_launch_counts(name, T):
    dev = torch.device("cuda", torch.cuda.current_device())
    s = bench.Setup(name, T, 0, dev)
    s.permute()
    torch.cuda.synchronize()
    kernels, nodes = kernel_nodes(s.permute)
    assert kernels == nodes == s.launches_per_permute(), (kernels, nodes)
    kernels, nodes = kernel_nodes(s.unpermute)
    assert kernels == nodes == 1


@pytest.mark.parametrize("T", [128, 256, 257, 4096])
def test_quant_permute_launch_counts(T):
    dev = torch.device("cuda", torch.cuda.current_device())
    s = bench.Setup("dsv3", T, 0, dev)
    s.enable_quant(dev)
    s.permute_quant()
    torch.cuda.synchronize()
    kernels, nodes = kernel_nodes(s.permute_quant)
    assert kernels == nodes == s.launches_per_permute(quant=True), (kernels, nodes)
