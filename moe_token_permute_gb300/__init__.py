"""GB300 (sm_103a) MoE token permute / unpermute behind a C ABI.

The Python functions below carry the names of the C entry points declared in
include/moe_permute.h and only marshal torch tensors into pointers and sizes;
all work runs in libmoe_permute.so.  Every output buffer and the workspace are
supplied by the caller, so no call allocates (vLLM PR #43014 digest,
"implementation breakdown": scratch allocated once and reused).
``MoEPermuteScratch`` allocates such a set of buffers once, up front.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import _binding as _b
from ._binding import (MOE_FLAG_BARRIER_TIMEOUT, MOE_FLAG_CAPACITY_OVERFLOW,  # noqa: F401
                       MOE_FLAG_ID_OUT_OF_RANGE, MOE_FLAG_INV_OUT_OF_RANGE,
                       MOE_FLAG_MAP_OUT_OF_RANGE, MOE_MAX_LOCAL_EXPERTS, MOE_MAX_TOPK,
                       MoeError, library_path)

_DTYPES = {
    torch.bfloat16: _b.MOE_DTYPE_BF16,
    torch.float16: _b.MOE_DTYPE_FP16,
    torch.float8_e4m3fn: _b.MOE_DTYPE_FP8_E4M3,
    torch.float8_e5m2: _b.MOE_DTYPE_FP8_E5M2,
    torch.float32: _b.MOE_DTYPE_FP32,
}
_INDEX = {torch.int32: _b.MOE_INDEX_INT32, torch.int64: _b.MOE_INDEX_INT64}


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor (the library writes in place)")
    return t.data_ptr()


def _need(t, n, what):
    """The C entry points take bare pointers, so a buffer too small for the
    call would be written or read out of bounds on the device: refuse it
    here, before any pointer is taken."""
    if t is not None and t.numel() < n:
        raise ValueError(f"{what} holds {t.numel()} elements; this call needs {n}")


def _need_bytes(t, n, what):
    if t is not None and t.numel() * t.element_size() < n:
        raise ValueError(f"{what} holds {t.numel() * t.element_size()} bytes; this call needs {n}")


def _need_rows(t, T, what):
    if t is not None and (t.dim() != 2 or t.shape[0] < T):
        raise ValueError(f"{what} must be 2-D with at least {T} rows (one per token)")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def moe_permute_supported(device: int | None = None) -> bool:
    if device is None:
        device = torch.cuda.current_device()
    return _b.lib().moe_permute_supported(int(device)) == 1


def moe_permute_workspace_size(max_tokens: int, topk: int, num_experts: int) -> int:
    n = _b.lib().moe_permute_workspace_size(int(max_tokens), int(topk), int(num_experts))
    if n == 0:
        raise ValueError("invalid workspace size arguments")
    return int(n)


def moe_permute_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    _b.check("moe_permute_workspace_init",
             _b.lib().moe_permute_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                                 _stream(stream)))


def moe_permute(hidden_states, topk_ids, expert_first_token_offset, permuted_idx,
                inv_permuted_idx, workspace, *, num_experts, num_local_experts=None,
                expert_map=None, hidden_scales=None, permuted_hidden_states=None,
                permuted_scales=None, stream=None) -> None:
    """Permute in place into the given buffers (see include/moe_permute.h).

    hidden_states [T,H] (None for a metadata-only call), topk_ids [T,K] int32
    or int64, expert_first_token_offset int64 [E_local+1], permuted_idx and
    inv_permuted_idx int32 [T*K], workspace uint8 (moe_permute_workspace_size),
    permuted_hidden_states [T*K,H] or None, hidden_scales [T,S] fp32 and
    permuted_scales [T*K,S] fp32 or both None.
    """
    T, K = topk_ids.shape
    if num_local_experts is None:
        num_local_experts = num_experts
    _need_rows(hidden_states, T, "hidden_states")
    _need_rows(hidden_scales, T, "hidden_scales")
    if hidden_states is not None:
        H = hidden_states.shape[1]
        dt = _DTYPES[hidden_states.dtype]
        _need_bytes(permuted_hidden_states, T * K * H * hidden_states.element_size(),
                    "permuted_hidden_states")
    else:
        H, dt = 1, _b.MOE_DTYPE_BF16
    scale_cols = hidden_scales.shape[1] if hidden_scales is not None else 0
    _need(permuted_scales, T * K * scale_cols, "permuted_scales")
    _need(expert_first_token_offset, num_local_experts + 1, "expert_first_token_offset")
    _need(permuted_idx, T * K, "permuted_idx")
    _need(inv_permuted_idx, T * K, "inv_permuted_idx")
    _need(expert_map, num_experts, "expert_map")
    _b.check("moe_permute", _b.lib().moe_permute(
        _ptr(hidden_states), dt, _ptr(hidden_scales), scale_cols,
        _ptr(topk_ids), _INDEX[topk_ids.dtype], _ptr(expert_map),
        T, H, K, num_experts, num_local_experts,
        _ptr(permuted_hidden_states), _ptr(permuted_scales),
        _ptr(expert_first_token_offset), _ptr(permuted_idx), _ptr(inv_permuted_idx),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_permute_batched(hidden_states, topk_ids, expert_num_tokens, inv_permuted_idx, workspace,
                        *, num_experts, max_rows_per_expert, num_local_experts=None,
                        expert_map=None, hidden_scales=None, batched_hidden_states=None,
                        batched_scales=None, stream=None) -> None:
    """Permute into the batched layout (see include/moe_permute.h):
    batched_hidden_states [E_local * M, H] (or [E_local, M, H]),
    expert_num_tokens int32 [E_local], inv_permuted_idx int32 [T*K] holding
    slots e*M + j."""
    T, K = topk_ids.shape
    if num_local_experts is None:
        num_local_experts = num_experts
    slots = num_local_experts * int(max_rows_per_expert)
    _need_rows(hidden_states, T, "hidden_states")
    _need_rows(hidden_scales, T, "hidden_scales")
    if hidden_states is not None:
        H = hidden_states.shape[1]
        dt = _DTYPES[hidden_states.dtype]
        _need_bytes(batched_hidden_states, slots * H * hidden_states.element_size(),
                    "batched_hidden_states")
    else:
        H, dt = 1, _b.MOE_DTYPE_BF16
    scale_cols = hidden_scales.shape[1] if hidden_scales is not None else 0
    _need(batched_scales, slots * scale_cols, "batched_scales")
    _need(expert_num_tokens, num_local_experts, "expert_num_tokens")
    _need(inv_permuted_idx, T * K, "inv_permuted_idx")
    _need(expert_map, num_experts, "expert_map")
    _b.check("moe_permute_batched", _b.lib().moe_permute_batched(
        _ptr(hidden_states), dt, _ptr(hidden_scales), scale_cols,
        _ptr(topk_ids), _INDEX[topk_ids.dtype], _ptr(expert_map),
        T, H, K, num_experts, num_local_experts, int(max_rows_per_expert),
        _ptr(batched_hidden_states), _ptr(batched_scales), _ptr(expert_num_tokens),
        _ptr(inv_permuted_idx), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_permute_quant_fp8(hidden_states, topk_ids, expert_first_token_offset, permuted_idx,
                          inv_permuted_idx, workspace, permuted_codes, permuted_scales, *,
                          num_experts, num_local_experts=None, expert_map=None,
                          stream=None) -> None:
    """Permute bf16 rows and quantise them to fp8 e4m3 on the way (see
    include/moe_permute.h): permuted_codes [T*K, H] float8_e4m3fn,
    permuted_scales [T*K, H/128] float32."""
    T, K = topk_ids.shape
    if hidden_states.dtype != torch.bfloat16:
        raise ValueError("moe_permute_quant_fp8 takes bf16 hidden_states")
    if permuted_codes.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise ValueError("permuted_codes must be float8_e4m3fn (or raw uint8)")
    if num_local_experts is None:
        num_local_experts = num_experts
    _need_rows(hidden_states, T, "hidden_states")
    H = hidden_states.shape[1]
    _need_bytes(permuted_codes, T * K * H, "permuted_codes")
    _need(permuted_scales, T * K * (H // _b.MOE_QUANT_GROUP), "permuted_scales")
    _need(expert_first_token_offset, num_local_experts + 1, "expert_first_token_offset")
    _need(permuted_idx, T * K, "permuted_idx")
    _need(inv_permuted_idx, T * K, "inv_permuted_idx")
    _need(expert_map, num_experts, "expert_map")
    _b.check("moe_permute_quant_fp8", _b.lib().moe_permute_quant_fp8(
        _ptr(hidden_states), _ptr(topk_ids), _INDEX[topk_ids.dtype], _ptr(expert_map),
        T, hidden_states.shape[1], K, num_experts, num_local_experts,
        _ptr(permuted_codes), _ptr(permuted_scales), _ptr(expert_first_token_offset),
        _ptr(permuted_idx), _ptr(inv_permuted_idx), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_unpermute(permuted_rows, topk_weights, inv_permuted_idx, out, *, workspace=None,
                  stream=None) -> None:
    """out[t] = bf16(sum_k w[t,k] * permuted_rows[inv[t*K+k]]) in place.

    permuted_rows bf16 [num_rows,H], topk_weights fp32 [T,K], inv_permuted_idx
    int32 [T*K], out bf16 [T,H]; workspace optional (status word only).
    """
    T, K = topk_weights.shape
    H = out.shape[1]
    if permuted_rows.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("moe_unpermute takes bf16 rows and writes bf16")
    if topk_weights.dtype != torch.float32 or inv_permuted_idx.dtype != torch.int32:
        raise ValueError("topk_weights must be float32 and inv_permuted_idx int32")
    if permuted_rows.shape[1] != H:
        raise ValueError("hidden size mismatch between rows and out")
    _need_rows(out, T, "out")
    _need(inv_permuted_idx, T * K, "inv_permuted_idx")
    _b.check("moe_unpermute", _b.lib().moe_unpermute(
        _ptr(permuted_rows), permuted_rows.shape[0], _ptr(topk_weights),
        _ptr(inv_permuted_idx), T, H, K, _ptr(out), _ptr(workspace), _stream(stream)))


def moe_read_status(workspace, stream=None) -> int:
    """OR of the MOE_FLAG_* bits raised since the last clear (syncs the stream)."""
    import ctypes
    v = ctypes.c_uint32(0)
    _b.check("moe_read_status", _b.lib().moe_read_status(_ptr(workspace), ctypes.byref(v),
                                                        _stream(stream)))
    return int(v.value)


def moe_clear_status(workspace, stream=None) -> None:
    _b.check("moe_clear_status", _b.lib().moe_clear_status(_ptr(workspace), _stream(stream)))


def moe_permute_read_status(workspace, dst, *, clear_after_read=False, stream=None) -> None:
    """Enqueue a copy of the status word into dst (a 1-element int32/uint32
    tensor on the device, or in pinned host memory) and optionally clear the
    word; asynchronous and capturable into a CUDA graph."""
    if dst.dtype.is_floating_point or dst.element_size() != 4 or dst.numel() < 1:
        raise ValueError("dst must hold at least one 32-bit integer")
    if not dst.is_contiguous():
        raise ValueError("expected a contiguous tensor (the library writes in place)")
    if not dst.is_cuda and not dst.is_pinned():
        raise ValueError("dst must be device memory or pinned host memory")
    _b.check("moe_permute_read_status", _b.lib().moe_permute_read_status(
        _ptr(workspace), dst.data_ptr(), 1 if clear_after_read else 0, _stream(stream)))


@dataclass
class MoEPermuteScratch:
    """Buffers for repeated permutes, allocated once (vLLM PR #43014 digest,
    "key source excerpts": MoEPermuteScratch.__post_init__, validate,
    token_expert_indices_view, prepare_topk_ids).

    Holds the workspace and the metadata buffers for up to max_num_tokens
    tokens, plus permuted hidden (and fp8 scale) rows when hidden_size is
    given, the unpermute output [max_num_tokens, hidden_size] bf16, and, when
    max_rows_per_expert is given, the batched layout's buffers.  Every method
    validates its inputs against these sizes and writes into views of the same
    storage on every call: nothing is allocated after construction.

    The digest's sort workspace, sorted-row and int32-cast buffers have no
    counterpart: the routing is a counting sort whose whole scratch is the
    library's workspace, and int64 ids are read natively.
    """
    max_num_tokens: int
    topk: int
    num_experts: int
    num_local_experts: int
    device: torch.device
    hidden_size: int | None = None
    hidden_dtype: torch.dtype | None = None
    scale_cols: int = 0
    max_rows_per_expert: int | None = None
    token_expert_indices: torch.Tensor = field(init=False)
    workspace: torch.Tensor = field(init=False)
    expert_first_token_offset: torch.Tensor = field(init=False)
    permuted_idx: torch.Tensor = field(init=False)
    inv_permuted_idx: torch.Tensor = field(init=False)
    permuted_hidden_states: torch.Tensor | None = field(init=False, default=None)
    permuted_scales: torch.Tensor | None = field(init=False, default=None)
    unpermuted: torch.Tensor | None = field(init=False, default=None)
    expert_num_tokens: torch.Tensor | None = field(init=False, default=None)
    batched_hidden_states: torch.Tensor | None = field(init=False, default=None)
    batched_scales: torch.Tensor | None = field(init=False, default=None)

    def __post_init__(self):
        dev = torch.device(self.device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        rows = self.max_num_tokens * self.topk
        if not moe_permute_supported(dev.index if dev.index is not None else None):
            raise MoeError("MoEPermuteScratch: the current device is not an sm_103 GPU")
        nbytes = moe_permute_workspace_size(self.max_num_tokens, self.topk, self.num_experts)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        moe_permute_workspace_init(self.workspace)
        # r = t * topk + k; stored only so that token_expert_indices_view can
        # hand out the digest's [T, topk] view (the kernels compute r).
        self.token_expert_indices = torch.arange(rows, dtype=torch.int32, device=dev)
        self.expert_first_token_offset = torch.empty(self.num_local_experts + 1,
                                                     dtype=torch.int64, device=dev)
        self.permuted_idx = torch.empty(rows, dtype=torch.int32, device=dev)
        self.inv_permuted_idx = torch.empty(rows, dtype=torch.int32, device=dev)
        if self.hidden_size is not None:
            self.permuted_hidden_states = torch.empty(rows, self.hidden_size,
                                                      dtype=self.hidden_dtype, device=dev)
            if self.scale_cols:
                self.permuted_scales = torch.empty(rows, self.scale_cols,
                                                   dtype=torch.float32, device=dev)
            self.unpermuted = torch.empty(self.max_num_tokens, self.hidden_size,
                                          dtype=torch.bfloat16, device=dev)
        if self.max_rows_per_expert is not None:
            slots = self.num_local_experts * int(self.max_rows_per_expert)
            self.expert_num_tokens = torch.empty(self.num_local_experts, dtype=torch.int32,
                                                 device=dev)
            if self.hidden_size is not None:
                self.batched_hidden_states = torch.empty(slots, self.hidden_size,
                                                         dtype=self.hidden_dtype, device=dev)
                if self.scale_cols:
                    self.batched_scales = torch.empty(slots, self.scale_cols,
                                                      dtype=torch.float32, device=dev)

    def validate(self, hidden_states, topk_ids, hidden_scales=None):
        """Inputs must fit the sizes this scratch was built for."""
        n_token = topk_ids.shape[0]
        if topk_ids.device != self.device:
            raise ValueError("topk_ids is not on the scratch's device")
        if n_token > self.max_num_tokens:
            raise ValueError(f"{n_token} tokens > max_num_tokens={self.max_num_tokens}")
        if topk_ids.dim() != 2 or topk_ids.shape[1] != self.topk:
            raise ValueError("topk mismatch")
        if hidden_states is not None:
            if hidden_states.device != self.device:
                raise ValueError("hidden_states is not on the scratch's device")
            if hidden_states.shape[0] != n_token:
                raise ValueError("hidden_states / topk_ids token count mismatch")
            if self.hidden_size is not None and (hidden_states.shape[1] != self.hidden_size
                                                 or hidden_states.dtype != self.hidden_dtype):
                raise ValueError("hidden size / dtype mismatch")
        if hidden_states is not None and self.hidden_size is not None and \
                (hidden_scales is not None) != bool(self.scale_cols):
            raise ValueError("scales given iff the scratch holds scale rows")
        if hidden_scales is not None and tuple(hidden_scales.shape) != (n_token, self.scale_cols):
            raise ValueError(f"hidden_scales must be [{n_token}, {self.scale_cols}]")

    def token_expert_indices_view(self, n_token: int) -> torch.Tensor:
        """The expanded row ids r = t * topk + k of n_token tokens, as [n_token, topk]."""
        if n_token > self.max_num_tokens:
            raise ValueError(f"{n_token} tokens > max_num_tokens={self.max_num_tokens}")
        return self.token_expert_indices[:n_token * self.topk].view(n_token, self.topk)

    def prepare_topk_ids(self, topk_ids: torch.Tensor) -> torch.Tensor:
        """The ids as the kernels take them: int32 and int64 are both read
        natively, so this is the tensor itself (no cast, no copy)."""
        if topk_ids.dtype not in _INDEX:
            raise ValueError("topk_ids must be int32 or int64")
        return topk_ids

    def _rows(self, topk_ids):
        return topk_ids.shape[0] * self.topk

    def permute(self, hidden_states, topk_ids, *, expert_map=None, hidden_scales=None,
                stream=None):
        """Permute into this scratch; returns views sized for this call."""
        self.validate(hidden_states, topk_ids, hidden_scales)
        n = self._rows(topk_ids)
        ph = None
        ps = None
        if self.permuted_hidden_states is not None and hidden_states is not None:
            ph = self.permuted_hidden_states[:n]
            if hidden_scales is not None:
                ps = self.permuted_scales[:n]
        moe_permute(hidden_states, self.prepare_topk_ids(topk_ids),
                    self.expert_first_token_offset,
                    self.permuted_idx[:n], self.inv_permuted_idx[:n], self.workspace,
                    num_experts=self.num_experts, num_local_experts=self.num_local_experts,
                    expert_map=expert_map, hidden_scales=hidden_scales,
                    permuted_hidden_states=ph, permuted_scales=ps, stream=stream)
        return dict(permuted_hidden_states=ph, permuted_scales=ps,
                    expert_first_token_offset=self.expert_first_token_offset,
                    permuted_idx=self.permuted_idx[:n], inv_permuted_idx=self.inv_permuted_idx[:n])

    def permute_quant_fp8(self, hidden_states, topk_ids, *, expert_map=None, stream=None):
        """Permute bf16 rows and quantise them to fp8 e4m3 on the way, into
        this scratch's rows and scales.  The scratch must have been built with
        hidden_dtype=torch.float8_e4m3fn and scale_cols = hidden_size / 128."""
        if self.hidden_dtype != torch.float8_e4m3fn or self.hidden_size is None or \
                self.scale_cols != self.hidden_size // _b.MOE_QUANT_GROUP:
            raise ValueError("permute_quant_fp8 needs a scratch of float8_e4m3fn rows with "
                             "hidden_size / 128 scale columns")
        if hidden_states.dtype != torch.bfloat16 or hidden_states.device != self.device:
            raise ValueError("permute_quant_fp8 takes bf16 hidden_states on the scratch's device")
        if hidden_states.shape != (topk_ids.shape[0], self.hidden_size):
            raise ValueError(f"hidden_states must be [{topk_ids.shape[0]}, {self.hidden_size}]")
        self.validate(None, topk_ids)
        n = self._rows(topk_ids)
        codes = self.permuted_hidden_states[:n]
        scales = self.permuted_scales[:n]
        moe_permute_quant_fp8(hidden_states, self.prepare_topk_ids(topk_ids),
                              self.expert_first_token_offset, self.permuted_idx[:n],
                              self.inv_permuted_idx[:n], self.workspace, codes, scales,
                              num_experts=self.num_experts,
                              num_local_experts=self.num_local_experts, expert_map=expert_map,
                              stream=stream)
        return dict(permuted_hidden_states=codes, permuted_scales=scales,
                    expert_first_token_offset=self.expert_first_token_offset,
                    permuted_idx=self.permuted_idx[:n], inv_permuted_idx=self.inv_permuted_idx[:n])

    def permute_batched(self, hidden_states, topk_ids, *, expert_map=None, hidden_scales=None,
                        stream=None):
        """Permute into this scratch's batched [E_local, M, H] layout
        (M = max_rows_per_expert); inv_permuted_idx then holds slots e*M + j."""
        if self.max_rows_per_expert is None:
            raise ValueError("permute_batched needs a scratch built with max_rows_per_expert")
        self.validate(hidden_states, topk_ids, hidden_scales)
        n = self._rows(topk_ids)
        bh = self.batched_hidden_states if hidden_states is not None else None
        bs = self.batched_scales if hidden_states is not None else None
        moe_permute_batched(hidden_states, self.prepare_topk_ids(topk_ids),
                            self.expert_num_tokens, self.inv_permuted_idx[:n], self.workspace,
                            num_experts=self.num_experts,
                            max_rows_per_expert=self.max_rows_per_expert,
                            num_local_experts=self.num_local_experts, expert_map=expert_map,
                            hidden_scales=hidden_scales, batched_hidden_states=bh,
                            batched_scales=bs, stream=stream)
        M = int(self.max_rows_per_expert)
        return dict(batched_hidden_states=None if bh is None
                    else bh.view(self.num_local_experts, M, self.hidden_size),
                    batched_scales=None if bs is None
                    else bs.view(self.num_local_experts, M, self.scale_cols),
                    expert_num_tokens=self.expert_num_tokens,
                    inv_permuted_idx=self.inv_permuted_idx[:n])

    def unpermute(self, permuted_rows, topk_weights, *, out=None, stream=None):
        """Reduce the grouped GEMM's output rows back to tokens through the
        inverse map the last permute of this scratch wrote (contiguous or
        batched).  Writes into `out` if given, else into this scratch's
        unpermute buffer; returns the [T, H] result."""
        T = topk_weights.shape[0]
        if T > self.max_num_tokens or topk_weights.dim() != 2 or topk_weights.shape[1] != self.topk:
            raise ValueError("topk_weights must be [T, topk] with T <= max_num_tokens")
        if out is None:
            if self.unpermuted is None or permuted_rows.shape[1] != self.hidden_size:
                raise ValueError("no unpermute buffer of this hidden size: pass out=")
            out = self.unpermuted[:T]
        moe_unpermute(permuted_rows, topk_weights, self.inv_permuted_idx[:T * self.topk], out,
                      workspace=self.workspace, stream=stream)
        return out

    def read_status(self, stream=None) -> int:
        """OR of the MOE_FLAG_* bits raised since the last clear (syncs the stream)."""
        return moe_read_status(self.workspace, stream)

    def clear_status(self, stream=None) -> None:
        moe_clear_status(self.workspace, stream)
