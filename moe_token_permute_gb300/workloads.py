"""Seeded synthetic inputs for the MoE permute / unpermute path.

This module only draws random inputs; it holds none of the permute or
unpermute arithmetic and imports neither the CUDA binding nor the oracle, so
both sides of every parity test can take their inputs from here.

The shapes are those of the MoE layers of the models the pages evaluate or
name (vLLM PR #19636 lm-eval runs: Qwen3-30B-A3B, DeepSeek-Coder-V2-Lite),
plus Mixtral-8x7B and DeepSeek-V3 layers.  No public dataset is used: routing
is drawn from a uniform or Zipf expert popularity as stated per workload.

Draw order for one (workload, T), from a generator freshly seeded with
``seed``: hidden, topk_ids, topk_weights, expert_map, expert-output rows (the
rows come last so that skipping them leaves every other input unchanged).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

FP8_MAX = 448.0  # largest finite float8_e4m3fn value
FP8_BLOCK = 128  # columns per activation scale


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    E: int
    K: int
    hidden_dtype: str          # "bf16" or "fp8"
    routing: str               # "uniform" or "zipf"
    zipf_s: float = 0.0
    E_local: int | None = None  # set => an expert_map marks E_local experts local
    T_sweep: tuple = field(default_factory=tuple)

    @property
    def e_local(self) -> int:
        return self.E if self.E_local is None else self.E_local


WORKLOADS = {
    "tiny": Workload("tiny", H=128, E=8, K=2, hidden_dtype="bf16",
                     routing="uniform", T_sweep=(16,)),
    "mixtral": Workload("mixtral", H=4096, E=8, K=2, hidden_dtype="bf16",
                        routing="uniform", T_sweep=(1, 32, 512, 4096, 16384)),
    "qwen3": Workload("qwen3", H=2048, E=128, K=8, hidden_dtype="bf16",
                      routing="zipf", zipf_s=1.2,
                      T_sweep=(1, 64, 1024, 8192, 16384)),
    "dsv2lite": Workload("dsv2lite", H=2048, E=64, K=6, hidden_dtype="bf16",
                         routing="uniform", E_local=16, T_sweep=(1, 256, 8192)),
    "dsv3": Workload("dsv3", H=7168, E=256, K=8, hidden_dtype="fp8",
                     routing="zipf", zipf_s=1.0, T_sweep=(1, 128, 4096, 32768)),
}


def _generator(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_hidden(wl: Workload, T: int, g, device):
    """bf16 N(0,1) [T,H]; or fp8 e4m3 codes [T,H] with fp32 scales [T,H/128].

    The fp8 input is prepared the usual way for block-scaled activations:
    scale = amax(block) / 448 (1 for an all-zero block), code = e4m3(x/scale).
    Permute only copies these bytes, so the recipe does not affect parity.
    """
    if wl.hidden_dtype == "bf16":
        return torch.randn(T, wl.H, generator=g, device=device,
                           dtype=torch.bfloat16), None
    x = torch.randn(T, wl.H // FP8_BLOCK, FP8_BLOCK, generator=g, device=device)
    amax = x.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    codes = (x / scale).to(torch.float8_e4m3fn).reshape(T, wl.H)
    return codes, scale.reshape(T, wl.H // FP8_BLOCK).contiguous()


def draw_topk_ids(wl: Workload, T: int, g, device):
    """int32 [T,K]: K distinct experts per token."""
    if wl.routing == "uniform":
        u = torch.rand(T, wl.E, generator=g, device=device)
        return u.argsort(dim=1)[:, :wl.K].to(torch.int32).contiguous()
    order = torch.randperm(wl.E, generator=g, device=device)
    rank = torch.arange(1, wl.E + 1, device=device, dtype=torch.float64)
    pop = torch.empty(wl.E, dtype=torch.float64, device=device)
    pop[order] = rank.pow(-wl.zipf_s)
    pop = (pop / pop.sum()).to(torch.float32)
    if T == 0:
        return torch.empty(0, wl.K, dtype=torch.int32, device=device)
    ids = torch.multinomial(pop.expand(T, wl.E), wl.K, replacement=False,
                            generator=g)
    return ids.to(torch.int32).contiguous()


def draw_topk_weights(wl: Workload, T: int, g, device):
    """fp32 [T,K] softmax of N(0,1) logits."""
    logits = torch.randn(T, wl.K, generator=g, device=device)
    return torch.softmax(logits, dim=-1).contiguous()


def draw_expert_rows(wl: Workload, T: int, g, device):
    """bf16 N(0,1) [T*K, H]: stands in for the grouped-GEMM output."""
    return torch.randn(T * wl.K, wl.H, generator=g, device=device,
                       dtype=torch.bfloat16)


def draw_expert_map(wl: Workload, g, device):
    """int32 [E]: a seeded random E_local experts get local ids 0..E_local-1
    in ascending global-id order, the rest -1.  None without a map."""
    if wl.E_local is None:
        return None
    chosen = torch.randperm(wl.E, generator=g, device=device)[:wl.E_local]
    chosen, _ = chosen.sort()
    m = torch.full((wl.E,), -1, dtype=torch.int32, device=device)
    m[chosen] = torch.arange(wl.E_local, dtype=torch.int32, device=device)
    return m


def make_inputs(wl: Workload | str, T: int, seed: int = 0, device="cpu",
                with_rows: bool = True):
    """All inputs of one (workload, T) in the fixed draw order.

    Returns a dict: hidden, scales (fp8 only, else None), topk_ids int32,
    topk_weights fp32, rows (bf16 [T*K,H] or None), expert_map (or None),
    plus the workload.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    g = _generator(device, seed)
    hidden, scales = draw_hidden(wl, T, g, device)
    ids = draw_topk_ids(wl, T, g, device)
    weights = draw_topk_weights(wl, T, g, device)
    emap = draw_expert_map(wl, g, device)
    rows = draw_expert_rows(wl, T, g, device) if with_rows else None
    return dict(wl=wl, T=T, hidden=hidden, scales=scales, topk_ids=ids,
                topk_weights=weights, rows=rows, expert_map=emap)
