"""Benchmark of the MoE token permute -> unpermute path on GB300.

One step = moe_permute (routing metadata + row gather) followed by
moe_unpermute (weighted top-k reduce) over one batch of a Mixtral-8x7B-shaped
MoE layer (T=16384 tokens, H=4096, E=8, top-2, bf16), through the C ABI.
The metric is HBM throughput: algorithmic bytes the step must move divided by
its device time, in GB/s, with the fraction of the measured HBM peak.  The
per-op numbers, the token-count sweep over every workload shape and the T=1
latencies come in the same JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--no-sweep] [--no-cpu-baseline]

Multi-GPU (torchrun): every rank runs the same step on its own batch (the
path has no exchange step; weak scaling); timing is max over ranks.
--impl reference: the CPU oracle, timed on the host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from moe_token_permute_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "permute/unpermute HBM GB/s (% of GB300 peak) and µs/call vs token count"
HEADLINE = ("mixtral", 16384)
WORKLOAD_NAMES = {"mixtral": "mixtral-8x7b-moe-layer", "qwen3": "qwen3-30b-a3b-moe-layer",
                  "dsv2lite": "deepseek-v2-lite-moe-layer-expert-map",
                  "dsv3": "deepseek-v3-moe-layer", "tiny": "tiny-moe-layer"}
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "moe_token_permute_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


# ------------------------------------------------------------ byte models ---
def routing_counts(ids: torch.Tensor, emap, E: int, K: int):
    """(T_v, N_v): tokens with >= 1 kept row, kept rows (host-side accounting)."""
    g = ids.long()
    ok = (g >= 0) & (g < E)
    if emap is not None:
        loc = torch.where(ok, emap.long()[g.clamp(0, E - 1)], torch.full_like(g, -1))
        ok = loc >= 0
    return int(ok.any(dim=1).sum()), int(ok.sum())


def permute_bytes(T, H, K, E_L, elem, scale_cols, Tv, Nv):
    """ids + source rows read once + K-fold row writes + both index maps + offsets."""
    rb = H * elem + scale_cols * 4
    return T * K * 4 + Tv * rb + Nv * rb + 2 * T * K * 4 + (E_L + 1) * 8


def gather_kernel_bytes(T, H, K, elem, scale_cols, Tv, Nv):
    rb = H * elem + scale_cols * 4
    return T * K * 4 + Tv * rb + Nv * rb


def quant_permute_bytes(T, H, K, E_L, Tv, Nv, group=128):
    """ids + bf16 source rows read once + fp8 codes and fp32 scales written to
    every kept row + both index maps + offsets."""
    return T * K * 4 + Tv * H * 2 + Nv * (H + (H // group) * 4) + 2 * T * K * 4 + (E_L + 1) * 8


def metadata_bytes(T, K, E_L):
    """Metadata-only permute: int32 ids + both index maps + offsets."""
    return T * K * 4 + 2 * T * K * 4 + (E_L + 1) * 8


def unpermute_bytes(T, H, K, Nv):
    """inv + weights + kept expert rows read + output written."""
    return 2 * T * K * 4 + Nv * H * 2 + T * H * 2


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """SM clock / throttle-reason samples via NVML (read-only queries)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.ok = False
        self.samples = []
        self.period = period_s
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return
            self.nv, self.h = nv, h
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except (OSError, AttributeError, RuntimeError):
            self.ok = False

    def _sample(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c))
        self._reasons(self.h, ctypes.byref(r))
        self.samples.append((int(c.value), int(r.value)))

    def _loop(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._sample()
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()
            self._sample()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b)
        return {"sm_mhz": float(statistics.median(mhz)), "sm_max_mhz": float(self.max_mhz),
                "reasons": reasons, "samples": len(mhz), "source": "nvml"}


# ---------------------------------------------------------------- helpers ---
def max_over_ranks(x_ms, dist, device):
    """The slowest rank's time (no-op with one process): every rank runs the
    same step on its own token batch, and the job is as fast as its slowest."""
    if dist is None:
        return x_ms
    t = torch.tensor([x_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world, bytes_per_rank_step, ms_per_step):
    """Whole-job throughput: each of `world` ranks moves bytes_per_rank_step
    per step, in the slowest rank's step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for r in rec.get("kernels", []):
        if r.get("kernel") == kernel and r.get("workload") == workload and \
                r.get("source_sha") == kernel_source_sha():
            return r.get("dram_bytes_per_launch")
    return None


class Setup:
    """Device buffers for one (workload, T): inputs, outputs, workspace."""

    def __init__(self, name, T, seed, dev):
        import moe_token_permute_gb300 as mp
        self.mp = mp
        inp = make_inputs(name, T, seed=seed, device=dev)
        wl = inp["wl"]
        self.wl, self.T = wl, T
        self.hidden, self.scales = inp["hidden"], inp["scales"]
        self.ids, self.w, self.rows, self.emap = (inp["topk_ids"], inp["topk_weights"],
                                                  inp["rows"], inp["expert_map"])
        R = T * wl.K
        self.offsets = torch.empty(wl.e_local + 1, dtype=torch.int64, device=dev)
        self.pidx = torch.empty(R, dtype=torch.int32, device=dev)
        self.inv = torch.empty(R, dtype=torch.int32, device=dev)
        self.ph = torch.empty(R, wl.H, dtype=self.hidden.dtype, device=dev)
        self.ps = None if self.scales is None else torch.empty(R, self.scales.shape[1],
                                                               dtype=torch.float32, device=dev)
        self.out = torch.empty(T, wl.H, dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(mp.moe_permute_workspace_size(T, wl.K, wl.E), dtype=torch.uint8,
                              device=dev)
        mp.moe_permute_workspace_init(self.ws)
        self.Tv, self.Nv = routing_counts(self.ids, self.emap, wl.E, wl.K)
        elem = self.hidden.element_size()
        sc = 0 if self.scales is None else self.scales.shape[1]
        self.pbytes = permute_bytes(T, wl.H, wl.K, wl.e_local, elem, sc, self.Tv, self.Nv)
        self.gbytes = gather_kernel_bytes(T, wl.H, wl.K, elem, sc, self.Tv, self.Nv)
        self.ubytes = unpermute_bytes(T, wl.H, wl.K, self.Nv)

    def enable_quant(self, dev):
        """bf16 rows of the same shape and fp8 outputs for quantise-on-permute."""
        g = torch.Generator(device=dev).manual_seed(1234)
        R = self.T * self.wl.K
        self.qhidden = torch.randn(self.T, self.wl.H, generator=g, device=dev,
                                   dtype=torch.bfloat16)
        self.qcodes = torch.empty(R, self.wl.H, dtype=torch.float8_e4m3fn, device=dev)
        self.qscales = torch.empty(R, self.wl.H // 128, dtype=torch.float32, device=dev)
        self.qbytes = quant_permute_bytes(self.T, self.wl.H, self.wl.K, self.wl.e_local,
                                          self.Tv, self.Nv)

    def enable_batched(self, dev, M):
        """Batched-layout outputs with capacity M per local expert."""
        self.bM = M
        self.bcounts = torch.empty(self.wl.e_local, dtype=torch.int32, device=dev)
        self.bhidden = torch.empty(self.wl.e_local * M, self.wl.H, dtype=self.hidden.dtype,
                                   device=dev)
        self.bscales = None if self.scales is None else torch.empty(
            self.wl.e_local * M, self.scales.shape[1], dtype=torch.float32, device=dev)
        # same bytes as the contiguous permute minus the permuted_idx writes
        self.bbytes = self.pbytes - self.T * self.wl.K * 4

    def permute_batched(self):
        self.mp.moe_permute_batched(self.hidden, self.ids, self.bcounts, self.inv, self.ws,
                                    num_experts=self.wl.E, num_local_experts=self.wl.e_local,
                                    max_rows_per_expert=self.bM, expert_map=self.emap,
                                    hidden_scales=self.scales, batched_hidden_states=self.bhidden,
                                    batched_scales=self.bscales)

    def permute_quant(self):
        self.mp.moe_permute_quant_fp8(self.qhidden, self.ids, self.offsets, self.pidx, self.inv,
                                      self.ws, self.qcodes, self.qscales, num_experts=self.wl.E,
                                      num_local_experts=self.wl.e_local, expert_map=self.emap)

    def permute_metadata(self):
        """Routing metadata only (no row gather): the consumer gathers rows itself."""
        self.mp.moe_permute(None, self.ids, self.offsets, self.pidx, self.inv, self.ws,
                            num_experts=self.wl.E, num_local_experts=self.wl.e_local,
                            expert_map=self.emap)

    def permute(self):
        self.mp.moe_permute(self.hidden, self.ids, self.offsets, self.pidx, self.inv, self.ws,
                            num_experts=self.wl.E, num_local_experts=self.wl.e_local,
                            expert_map=self.emap, hidden_scales=self.scales,
                            permuted_hidden_states=self.ph, permuted_scales=self.ps)

    def unpermute(self):
        self.mp.moe_unpermute(self.rows, self.w, self.inv, self.out, workspace=self.ws)

    def launches_per_permute(self, quant=False):
        """Kernels one moe_permute (or moe_permute_quant_fp8) call launches:
        one single-launch kernel up to 2048 expanded rows for
        moe_permute_quant_fp8, and up to 3072 (4096 with an expert map) for
        moe_permute; above that one for a permute with an expert map (the
        single-launch expert-map kernel: these buffers are 16-byte aligned and
        every workload's blocks fit it), else the routing grid plus the gather."""
        R = self.T * self.wl.K
        if R <= (2048 if quant else 4096 if self.emap is not None else 3072):
            return 1
        return 1 if (self.emap is not None and not quant) else 2

    def footprint(self):
        ts = [self.hidden, self.scales, self.ids, self.w, self.rows, self.emap, self.offsets,
              self.pidx, self.inv, self.ph, self.ps, self.out]
        return sum(t.numel() * t.element_size() for t in ts if t is not None)


class EndToEnd:
    """A step from pinned host memory to pinned host memory through the public
    API: every step copies its inputs in (hidden rows, ids, weights, the expert
    rows unpermute reads), runs moe_permute + moe_unpermute, and copies the
    output and the expert offsets out.

    serial_ms: everything on one stream, one step after another.
    pipelined_ms: a serving-style schedule over two device buffer sets.  Step
    i's inputs go in on a copy stream while step i-1 computes, its kernels run
    on a compute stream, and its results come out on a second copy stream; a
    set is refilled only once its previous step's kernels and copies out are
    done.  Same bytes, same calls."""

    def __init__(self, sets, do_permute, quant):
        self.sets, self.do_permute = sets, do_permute
        self.dev_in = [[st.qhidden if quant else st.hidden, st.ids, st.w, st.rows] for st in sets]
        s0 = sets[0]
        self.h_in = [t.cpu().pin_memory() for t in self.dev_in[0]]
        self.h_out = [torch.empty_like(s0.out, device="cpu").pin_memory(),
                      torch.empty_like(s0.offsets, device="cpu").pin_memory()]
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out)

    def _copy_in(self, j):
        for d, h in zip(self.dev_in[j], self.h_in):
            d.copy_(h, non_blocking=True)

    def _compute(self, j):
        st = self.sets[j]
        self.do_permute(st)
        st.unpermute()

    def _copy_out(self, j):
        st = self.sets[j]
        self.h_out[0].copy_(st.out, non_blocking=True)
        self.h_out[1].copy_(st.offsets, non_blocking=True)

    @staticmethod
    def _timed(fn, n, reps=3):
        """Median over `reps` timed runs of n steps (ms per step): one stall of
        the shared host or link does not decide the number."""
        times = []
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn(n)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) / n)
        return statistics.median(times)

    def serial_ms(self, n):
        def run(k):
            for _ in range(k):
                self._copy_in(0)
                self._compute(0)
                self._copy_out(0)
        run(3)
        return self._timed(run, n)

    def pipelined_ms(self, n):
        cur = torch.cuda.current_stream()
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        n_sets = len(self.sets)

        start = torch.cuda.Event()
        in_done = [torch.cuda.Event() for _ in range(n_sets)]
        cmp_done = [torch.cuda.Event() for _ in range(n_sets)]
        out_done = [torch.cuda.Event() for _ in range(n_sets)]

        def run(k):
            start.record(cur)
            for st in (s_in, s_cmp, s_out):
                st.wait_event(start)
            for i in range(k):
                j = i % n_sets
                if i >= n_sets:
                    s_in.wait_event(out_done[j])  # set j's previous step is fully done
                with torch.cuda.stream(s_in):
                    self._copy_in(j)
                in_done[j].record(s_in)
                s_cmp.wait_event(in_done[j])
                with torch.cuda.stream(s_cmp):
                    self._compute(j)
                cmp_done[j].record(s_cmp)
                s_out.wait_event(cmp_done[j])
                with torch.cuda.stream(s_out):
                    self._copy_out(j)
                out_done[j].record(s_out)
            for st in (s_in, s_cmp, s_out):
                cur.wait_stream(st)
        run(3)
        return self._timed(run, n)


L2_BYTES = 129 * 1024 * 1024


def timed_calls(fn, n, flush=None):
    """Mean device time (us) of fn over n calls, events around each call; the
    L2 flush (if any) runs between calls, outside the events."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        if flush is not None:
            flush()
        starts[i].record()
        fn()
        ends[i].record()
    torch.cuda.synchronize()
    return 1e3 * sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / n


def back_to_back_us(fns, n):
    """Mean device time (us) per call of n back-to-back calls cycling through
    fns (one per buffer set), one event pair around all of them."""
    for f in fns:
        f()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(n):
        fns[i % len(fns)]()
    b.record()
    torch.cuda.synchronize()
    return 1e3 * a.elapsed_time(b) / n


def graph_us(fns, n=100):
    """Per-call time from replaying a CUDA graph of n back-to-back calls."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in fns:
            f()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fns[i % len(fns)]()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return 1e3 * a.elapsed_time(b) / (reps * n)


def c_abi_latency(name, T, iters=300):
    """Per-call latency through the C ABI from a plain C program (no Python in
    the loop), medians in us: *_c_abi_issue_us = host time per call of
    back-to-back calls; *_c_abi_sync_us = one call plus a stream synchronise,
    after an idle gap; *_c_abi_device_us = CUDA events around one call after
    an idle gap; launch_floor_c_abi_* = the same for a call that enqueues one
    tiny kernel (num_tokens = 0), the floor of any call on this machine.
    Empty if the probe cannot be built or run."""
    from moe_token_permute_gb300 import build as cuda_build
    wl = WORKLOADS[name]
    fp8 = name == "dsv3"
    args = [wl.H, wl.E, wl.e_local, wl.K, 2 if fp8 else 0, wl.H // 128 if fp8 else 0, T, iters]
    try:
        exe = cuda_build.build_c_latency()
        outp = subprocess.run([exe] + [str(a) for a in args], capture_output=True, text=True,
                              timeout=120, check=True).stdout
        r = json.loads(outp.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError) as exc:
        print(f"c_abi_latency {name} T={T}: {exc}", file=sys.stderr)
        return {}
    return {f"{op}_c_abi_{kind}_us": r[f"{op}_{kind}_us"]
            for op in ("permute", "unpermute", "launch_floor") for kind in ("issue", "sync", "device")}


def sweep(dev, peak, flush):
    """Per (workload, T): permute and unpermute timed separately, rotating over
    enough buffer sets that the footprint is at least 3x the L2 size (or 64
    sets for the smallest batches).  *_us is the device time per call from
    replaying a CUDA graph of back-to-back calls (no Python launch cost);
    *_eager_us the same calls launched one by one from Python (1000 of them
    up to 64 tokens); at T = 1 also a
    single eager call after an L2 flush.  metadata_permute_us: the routing
    metadata alone (no row gather), a latency workload.  For the DeepSeek-V3 shape also
    quantise-on-permute from bf16 rows (quant_fp8_permute_*); for the Qwen3
    shape also the batched layout with capacity M = T (batched_permute_*)."""
    rows = []
    for name, wl in WORKLOADS.items():
        if name == "tiny":
            continue
        for T in wl.T_sweep:
            torch.cuda.nvtx.range_push(f"sweep {name} T={T}")
            first = Setup(name, T, seed=0, dev=dev)
            fp = first.footprint()
            n_sets = int(min(64, max(2, -(-3 * L2_BYTES // max(fp, 1)))))
            sets = [first] + [Setup(name, T, seed=i, dev=dev) for i in range(1, n_sets)]
            n = max(3 * n_sets, 30 if T >= 4096 else (1000 if T <= 64 else 200))
            n_graph = max(n_sets, 20 if T >= 4096 else 100)
            p_us = graph_us([s.permute for s in sets], n_graph)
            u_us = graph_us([s.unpermute for s in sets], n_graph)
            s0 = sets[0]
            rec = {"workload": name, "T": T, "sets": n_sets,
                   "permute_us": round(p_us, 2), "permute_GBps": round(s0.pbytes / p_us / 1e3, 1),
                   "permute_frac": round(s0.pbytes / p_us / 1e3 / peak, 4),
                   "unpermute_us": round(u_us, 2), "unpermute_GBps": round(s0.ubytes / u_us / 1e3, 1),
                   "unpermute_frac": round(s0.ubytes / u_us / 1e3 / peak, 4),
                   "permute_eager_us": round(back_to_back_us([s.permute for s in sets], n), 2),
                   "unpermute_eager_us": round(back_to_back_us([s.unpermute for s in sets], n), 2)}
            m_us = graph_us([s.permute_metadata for s in sets], n_graph)
            rec["metadata_permute_us"] = round(m_us, 2)
            rec["metadata_permute_GBps"] = round(
                metadata_bytes(T, s0.wl.K, s0.wl.e_local) / m_us / 1e3, 1)
            if name == "qwen3" and T >= 1024:
                for st in sets:
                    st.enable_batched(dev, T)
                b_us = graph_us([st.permute_batched for st in sets], n_graph)
                rec["batched_permute_us"] = round(b_us, 2)
                rec["batched_permute_GBps"] = round(s0.bbytes / b_us / 1e3, 1)
                rec["batched_permute_frac"] = round(s0.bbytes / b_us / 1e3 / peak, 4)
            if name == "dsv3":
                for st in sets:
                    st.enable_quant(dev)
                q_us = graph_us([st.permute_quant for st in sets], n_graph)
                rec["quant_fp8_permute_us"] = round(q_us, 2)
                rec["quant_fp8_permute_GBps"] = round(s0.qbytes / q_us / 1e3, 1)
                rec["quant_fp8_permute_frac"] = round(s0.qbytes / q_us / 1e3 / peak, 4)
            if T == 1:
                rec["permute_after_flush_us"] = round(timed_calls(s0.permute, 50, flush), 2)
                rec["unpermute_after_flush_us"] = round(timed_calls(s0.unpermute, 50, flush), 2)
                rec.update(c_abi_latency(name, T))
            rows.append(rec)
            del sets, first, s0
            torch.cuda.empty_cache()
            torch.cuda.nvtx.range_pop()
    return rows


# ------------------------------------------------------------- CPU oracle ---
class OracleStep:
    """The CPU oracle (permute with the row copy, then unpermute) on the
    headline workload's host inputs, optionally on its first T_sample tokens."""

    def __init__(self):
        import oracle
        self.oracle = oracle
        name, T = HEADLINE
        inp = make_inputs(name, T, seed=0)
        self.wl = inp["wl"]
        self.T = T
        self.ids_t = inp["topk_ids"]
        self.ids = inp["topk_ids"].numpy()
        self.hidden = inp["hidden"].view(torch.int16).numpy()
        self.rows = inp["rows"].view(torch.int16).numpy().view(np.uint16)
        self.w = inp["topk_weights"].numpy()

    def nbytes(self, Ts):
        wl = self.wl
        Tv, Nv = routing_counts(self.ids_t[:Ts], None, wl.E, wl.K)
        return permute_bytes(Ts, wl.H, wl.K, wl.e_local, 2, 0, Tv, Nv) + \
            unpermute_bytes(Ts, wl.H, wl.K, Nv)

    def run(self, Ts):
        """One step on the first Ts tokens; returns its wall time in seconds."""
        K = self.wl.K
        t0 = time.perf_counter()
        ref = self.oracle.permute(self.ids[:Ts], self.wl.E, hidden=self.hidden[:Ts])
        self.oracle.unpermute(self.rows[:Ts * K], self.w[:Ts], ref["inv_permuted_idx"])
        return time.perf_counter() - t0


def cpu_baseline(budget_s=12.0):
    """Repeat full-size oracle steps for about budget_s seconds of CPU work."""
    o = OracleStep()
    total, reps = 0.0, 0
    while total < budget_s:
        total += o.run(o.T)
        reps += 1
    per_step = total / reps
    return {"value": round(o.nbytes(o.T) / per_step / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"mixtral T={o.T} H=4096 E=8 K=2: {reps} full oracle permute+unpermute "
                      f"steps, {total:.1f} s of single-thread CPU work"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, single-threaded, on the
    headline workload; each step a sample of its first T_s tokens, sized so
    warm-up plus timed steps stay within about two minutes."""
    if rank != 0:
        return
    o = OracleStep()
    t1 = o.run(o.T)
    per_step_budget = 120.0 / (args.steps + args.warmup)
    Ts = max(1, min(o.T, int(o.T * per_step_budget / t1)))
    for _ in range(args.warmup):
        o.run(Ts)
    times = [o.run(Ts) for _ in range(args.steps)]
    step_s = sum(times) / len(times)
    value = o.nbytes(Ts) / step_s / 1e9
    sample = (f"mixtral-shaped layer (H=4096, E=8, K=2), first {Ts} of {o.T} tokens per step: "
              "one oracle permute (with row copy) + unpermute, single thread")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "mixtral-8x7b-moe-layer", "T": o.T, "T_sample": Ts,
                       "H": 4096, "E": 8, "K": 2},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- main ---
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=HEADLINE[0], choices=sorted(WORKLOADS),
                    help="layer shape of the timed step (default: the headline)")
    ap.add_argument("--tokens", type=int, default=HEADLINE[1], help="tokens per step")
    ap.add_argument("--quant", action="store_true",
                    help="permute bf16 rows with quantise-on-permute (fp8 e4m3 out)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import moe_token_permute_gb300 as mp
    mp._binding.lib()  # fails loudly if the CUDA library was not built
    if not mp.moe_permute_supported(local):
        raise SystemExit("this GPU is not an sm_103 device")

    peak, peak_kind = measured_peak()
    name, T = args.workload, args.tokens
    sets = [Setup(name, T, seed=rank * 2 + i, dev=dev) for i in range(2)]
    s0 = sets[0]
    if args.quant:
        for st in sets:
            st.enable_quant(dev)
    perm_bytes = s0.qbytes if args.quant else s0.pbytes
    step_bytes = perm_bytes + s0.ubytes
    launches_per_step = s0.launches_per_permute(args.quant) + 1

    def do_permute(s):
        if args.quant:
            s.permute_quant()
        else:
            s.permute()

    def step(i):
        s = sets[i % 2]
        do_permute(s)
        s.unpermute()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # The K steps are captured once into a CUDA graph, outside the timed region,
    # as a serving loop runs them: every call is stream-ordered and allocates
    # nothing, so it captures, and the graph keeps the programmatic-dependent-
    # launch edges between consecutive kernels.  Timed region: one replay of
    # that graph, i.e. exactly K steps, one event pair around it.
    n = args.steps
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(n):
            step(i)
    graph.replay()  # untimed first replay (graph upload)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk, torch.cuda.nvtx.range("timed steps"):
        start.record()
        graph.replay()
        end.record()
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    ms_per_step = total_ms / n
    value = job_gbs(world, step_bytes, ms_per_step)
    del graph

    # The same K steps launched one by one from Python, for comparison.
    torch.cuda.synchronize()
    start.record()
    for i in range(n):
        step(i)
    end.record()
    torch.cuda.synchronize()
    eager_ms_per_step = max_over_ranks(start.elapsed_time(end), dist, dev) / n

    # Per-op split and the duration of the dominant kernel (k_unpermute, one
    # launch per moe_unpermute call) for the roofline: the K calls of each op
    # captured into one CUDA graph per op (the two input sets alternate as in
    # the steps) and replayed with one event pair around each replay, so the
    # calls keep their back-to-back launch overlap as in the timed steps
    # (median of 3 replays).  The split with an event pair around every eager
    # call is kept as eager_us_per_call: each call then also pays its launch.
    def op_graph(fn):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap):
            for i in range(n):
                fn(sets[i % 2])
        g.replay()
        torch.cuda.synchronize()
        return g

    def replay_us(g, reps=3):
        times = []
        for _ in range(reps):
            start.record()
            g.replay()
            end.record()
            torch.cuda.synchronize()
            times.append(1e3 * start.elapsed_time(end) / n)
        return statistics.median(times)

    g_op = op_graph(do_permute)
    perm_us = max_over_ranks(replay_us(g_op) / 1e3, dist, dev) * 1e3
    g_op = op_graph(lambda st: st.unpermute())
    unp_us = max_over_ranks(replay_us(g_op) / 1e3, dist, dev) * 1e3
    del g_op
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        s = sets[i % 2]
        ev[i][0].record()
        do_permute(s)
        ev[i][1].record()
        s.unpermute()
        ev[i][2].record()
    torch.cuda.synchronize()
    perm_eager_us = 1e3 * sum(e[0].elapsed_time(e[1]) for e in ev) / n
    unp_eager_us = 1e3 * sum(e[1].elapsed_time(e[2]) for e in ev) / n

    # end to end: pinned host inputs in, result out, every step
    n_e2e = min(n, 50)
    e2e = EndToEnd(sets, do_permute, args.quant)
    with torch.cuda.nvtx.range("end to end, serial"):
        e2e_serial_ms = max_over_ranks(e2e.serial_ms(n_e2e), dist, dev)
    with torch.cuda.nvtx.range("end to end, pipelined"):
        e2e_ms = max_over_ranks(e2e.pipelined_ms(n_e2e), dist, dev)
    e2e_value = job_gbs(world, step_bytes, e2e_ms)
    h2d, d2h = e2e.h2d, e2e.d2h

    line = None
    if rank == 0:
        unp_gbs = s0.ubytes / unp_us / 1e3
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "timing": "one replay of a CUDA graph holding the K steps (captured before the "
                      "timed region); eager_*: the same K steps launched one by one",
            "eager_ms_per_step": round(eager_ms_per_step, 5),
            "eager_value": round(job_gbs(world, step_bytes, eager_ms_per_step), 1),
            "config": {"workload": WORKLOAD_NAMES[name] + ("-quant-fp8" if args.quant else ""),
                       "T": T, "H": s0.wl.H, "E": s0.wl.E, "E_local": s0.wl.e_local,
                       "K": s0.wl.K,
                       "routing": s0.wl.routing + (f" s={s0.wl.zipf_s}" if s0.wl.zipf_s else ""),
                       "parallelism": f"replicas x{world} (token batches, no collective)",
                       "l2": (f"inputs larger than L2: {step_bytes / 1e6:.0f} MB moved per step, "
                              "two input sets alternate") if step_bytes > L2_BYTES else
                             f"{step_bytes / 1e6:.0f} MB per step, two input sets alternate "
                             "(together within L2)"},
            "frac_of_peak": round(value / world / peak, 4),
            "peak_GBps": peak, "peak_kind": peak_kind,
            "bytes_per_step": step_bytes,
            "permute": {"us_per_call": round(perm_us, 2), "GBps": round(perm_bytes / perm_us / 1e3, 1),
                        "frac": round(perm_bytes / perm_us / 1e3 / peak, 4), "bytes": perm_bytes,
                        "launches": launches_per_step - 1,
                        "op": "moe_permute_quant_fp8" if args.quant else "moe_permute",
                        "eager_us_per_call": round(perm_eager_us, 2)},
            "unpermute": {"us_per_call": round(unp_us, 2), "GBps": round(unp_gbs, 1),
                          "frac": round(unp_gbs / peak, 4), "bytes": s0.ubytes, "launches": 1,
                          "eager_us_per_call": round(unp_eager_us, 2)},
            "roofline": {"kernel": "k_unpermute", "bound": "hbm", "achieved": round(unp_gbs, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(unp_gbs / peak, 4),
                         "peak_kind": peak_kind,
                         "traffic": ncu_traffic("k_unpermute", f"{name}-T{T}")},
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4), "steps": n_e2e,
                    "schedule": "pipelined: step i+1's host-to-device copy overlaps step i's "
                                "kernels and device-to-host copy (two device buffer sets, "
                                "separate copy and compute streams)",
                    "timing": "median of 3 timed runs of `steps` steps, each schedule",
                    "serial_ms_per_step": round(e2e_serial_ms, 4),
                    "serial_value": round(job_gbs(world, step_bytes, e2e_serial_ms), 1)},
            "gpu_launches": n * launches_per_step,
            "per_op_timing": "the K calls of each op replayed from one CUDA graph per op (inputs "
                             "alternating as in the steps), events around each replay; "
                             "eager_us_per_call: events around each eager call",
            "clocks": clk.summary(),
        }
    del e2e  # frees the pinned host copies before the sweep
    if rank == 0 and world == 1:
        flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        if not args.no_sweep:
            del sets, s0
            torch.cuda.empty_cache()
            line["sweep"] = sweep(dev, peak, flush=flush_buf.zero_)
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
