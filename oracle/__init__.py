"""CPU oracle for the MoE token permute / unpermute path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never loads it, and this package imports nothing from the product package.

The arithmetic lives in ``moe_oracle.c`` (plain single-threaded C, built with
``-ffp-contract=off``); this module only loads it and marshals numpy arrays.
``brute.py`` holds an independent pure-Python restatement used to pin the C
code on tiny inputs.

Definitions followed (see the header of ``moe_oracle.c`` for the readings):
  * vLLM PR #14568 "permute/unpermute kernel for moe optimization",
    description -- permute expands and orders tokens by expert; unpermute
    reduces the expanded rows back to tokens scaled by the top-k weights.
  * vLLM PR #43014 digest, section "key source excerpts" -- buffer names,
    shapes and dtypes of expert_first_token_offset, permuted_idx,
    inv_permuted_idx, permuted_hidden_states and token_expert_indices.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, invariants, hand-worked fixtures, closed forms, error bounds).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmoe_oracle.so")

FLAG_ID_RANGE = 1
FLAG_MAP_RANGE = 2
FLAG_INV_RANGE = 4
FLAG_CAPACITY = 16


def compile_source(src: str, out_path: str) -> str:
    """Compile one C source of the oracle into a shared object (gcc, plain C)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math",
                           "-std=c11", "-shared", "-fPIC", "-o", tmp, src])
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle with gcc if the shared object is missing or stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class OracleLib:
    """ctypes face of one compiled copy of the oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.oracle_permute.restype = ctypes.c_uint32
        lib.oracle_permute.argtypes = [P, I64, P, I64, P, ctypes.c_int, P, I64,
                                       I32, I32, I32, P, P, P, P, P]
        lib.oracle_unpermute.restype = ctypes.c_uint32
        lib.oracle_unpermute.argtypes = [P, I64, P, P, I64, I64, I32, P]
        lib.oracle_f32_to_bf16_rne.restype = None
        lib.oracle_f32_to_bf16_rne.argtypes = [P, I64, P]
        lib.oracle_permute_batched.restype = ctypes.c_uint32
        lib.oracle_permute_batched.argtypes = [P, I64, P, I64, P, ctypes.c_int, P, I64, I32,
                                               I32, I32, I64, P, P, P, P]
        lib.oracle_f32_to_e4m3.restype = None
        lib.oracle_f32_to_e4m3.argtypes = [P, I64, P]
        lib.oracle_quantize_fp8.restype = None
        lib.oracle_quantize_fp8.argtypes = [P, I64, I64, I64, P, P]
        self.lib = lib
        self.path = path

    def permute(self, topk_ids, E, *, expert_map=None, E_local=None,
                hidden=None, scales=None):
        return _permute(self.lib, topk_ids, E, expert_map, E_local, hidden, scales)

    def unpermute(self, rows_bf16_bits, topk_weights, inv_permuted_idx):
        return _unpermute(self.lib, rows_bf16_bits, topk_weights, inv_permuted_idx)

    def f32_to_bf16_rne(self, x):
        return _f32_to_bf16_rne(self.lib, x)

    def permute_batched(self, topk_ids, E, M, *, expert_map=None, E_local=None,
                        hidden=None, scales=None):
        """Batched layout: returns expert_num_tokens int32 [E_local],
        inv_permuted_idx int32 [T*K] (slot e*M+j or -1), batched_hidden
        [E_local*M, ...] and batched_scales (unused slots zero), flags."""
        topk_ids = np.ascontiguousarray(topk_ids)
        T, K = topk_ids.shape
        if expert_map is None:
            E_local = E if E_local is None else E_local
        else:
            expert_map = np.ascontiguousarray(expert_map, dtype=np.int32)
        cnt = np.zeros(E_local, np.int32)
        inv = np.zeros(T * K, np.int32)
        bh, row_bytes = None, 0
        if hidden is not None:
            hidden = np.ascontiguousarray(hidden)
            row_bytes = int(np.prod(hidden.shape[1:])) * hidden.itemsize
            bh = np.zeros((E_local * M,) + hidden.shape[1:], hidden.dtype)
        bs, scale_cols = None, 0
        if scales is not None:
            scales = np.ascontiguousarray(scales, dtype=np.float32)
            scale_cols = scales.shape[1]
            bs = np.zeros((E_local * M, scale_cols), np.float32)
        flags = self.lib.oracle_permute_batched(
            _ptr(hidden), row_bytes, _ptr(scales), scale_cols, _ptr(topk_ids),
            int(topk_ids.dtype == np.int64), _ptr(expert_map), T, K, E, E_local, M,
            _ptr(cnt), _ptr(inv), _ptr(bh), _ptr(bs))
        if flags == 0xFFFFFFFF:
            raise MemoryError("oracle_permute_batched: host allocation failed")
        return dict(expert_num_tokens=cnt, inv_permuted_idx=inv, batched_hidden=bh,
                    batched_scales=bs, flags=int(flags))

    def f32_to_e4m3(self, x):
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
        out = np.zeros(x.shape[0], np.uint8)
        self.lib.oracle_f32_to_e4m3(_ptr(x), x.shape[0], _ptr(out))
        return out

    def quantize_fp8(self, x_bf16_bits, group=128):
        """bf16 rows [T, H] (uint16 bits) -> (e4m3 codes uint8 [T, H],
        fp32 scales [T, H / group])."""
        x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
        T, H = x.shape
        assert H % group == 0
        codes = np.zeros((T, H), np.uint8)
        scales = np.zeros((T, H // group), np.float32)
        self.lib.oracle_quantize_fp8(_ptr(x), T, H, group, _ptr(codes), _ptr(scales))
        return codes, scales


_default = None


def _load() -> OracleLib:
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def permute(topk_ids, E, *, expert_map=None, E_local=None, hidden=None,
            scales=None):
    """Run the oracle permute (see ``_permute``)."""
    return _load().permute(topk_ids, E, expert_map=expert_map, E_local=E_local,
                           hidden=hidden, scales=scales)


def unpermute(rows_bf16_bits, topk_weights, inv_permuted_idx):
    """Run the oracle unpermute (see ``_unpermute``)."""
    return _load().unpermute(rows_bf16_bits, topk_weights, inv_permuted_idx)


def f32_to_bf16_rne(x):
    """The oracle's hand-written fp32 -> bf16 rounding, exposed for pinning."""
    return _load().f32_to_bf16_rne(x)


def permute_batched(topk_ids, E, M, **kw):
    """Batched-layout permute (see moe_oracle.c)."""
    return _load().permute_batched(topk_ids, E, M, **kw)


def f32_to_e4m3(x):
    """The oracle's hand-written fp32 -> e4m3 (satfinite, RNE), for pinning."""
    return _load().f32_to_e4m3(x)


def quantize_fp8(x_bf16_bits, group=128):
    """Per-token, per-group fp8 quantisation (see moe_oracle.c)."""
    return _load().quantize_fp8(x_bf16_bits, group)


def _permute(lib, topk_ids: np.ndarray, E: int, expert_map: np.ndarray | None,
             E_local: int | None, hidden: np.ndarray | None,
             scales: np.ndarray | None):
    """Oracle permute.

    topk_ids: [T, K] int32 or int64.  hidden: [T, ...] any dtype (rows are
    copied as bytes) or None.  scales: [T, S] float32 or None.
    Returns a dict with offsets int64 [E_local+1], permuted_idx int32 [T*K],
    inv_permuted_idx int32 [T*K], permuted_hidden (rows >= n_valid zero),
    permuted_scales, n_valid and flags.
    """
    topk_ids = np.ascontiguousarray(topk_ids)
    assert topk_ids.ndim == 2 and topk_ids.dtype in (np.int32, np.int64)
    T, K = topk_ids.shape
    if expert_map is None:
        E_local = E if E_local is None else E_local
        assert E_local == E
    else:
        expert_map = np.ascontiguousarray(expert_map, dtype=np.int32)
        assert expert_map.shape == (E,)
        assert E_local is not None
    R = T * K
    offsets = np.zeros(E_local + 1, np.int64)
    pidx = np.zeros(R, np.int32)
    inv = np.zeros(R, np.int32)
    row_bytes = 0
    ph = None
    if hidden is not None:
        hidden = np.ascontiguousarray(hidden)
        assert hidden.shape[0] == T
        row_bytes = hidden[0].nbytes if T > 0 else int(np.prod(hidden.shape[1:])) * hidden.itemsize
        ph = np.zeros((R,) + hidden.shape[1:], hidden.dtype)
    ps = None
    scale_cols = 0
    if scales is not None:
        scales = np.ascontiguousarray(scales, dtype=np.float32)
        assert scales.ndim == 2 and scales.shape[0] == T
        scale_cols = scales.shape[1]
        ps = np.zeros((R, scale_cols), np.float32)
    flags = lib.oracle_permute(_ptr(hidden), row_bytes, _ptr(scales), scale_cols,
                               _ptr(topk_ids), int(topk_ids.dtype == np.int64),
                               _ptr(expert_map), T, K, E, E_local,
                               _ptr(offsets), _ptr(pidx), _ptr(inv), _ptr(ph), _ptr(ps))
    if flags == 0xFFFFFFFF:
        raise MemoryError("oracle_permute: host allocation failed")
    return dict(offsets=offsets, permuted_idx=pidx, inv_permuted_idx=inv,
                permuted_hidden=ph, permuted_scales=ps,
                n_valid=int(offsets[-1]), flags=int(flags))


def _unpermute(lib, rows_bf16_bits: np.ndarray, topk_weights: np.ndarray,
               inv_permuted_idx: np.ndarray):
    """Oracle unpermute.

    rows_bf16_bits: [num_rows, H] uint16 (bf16 bit patterns).
    topk_weights: [T, K] float32.  inv_permuted_idx: [T*K] int32.
    Returns (out uint16 [T, H] bf16 bits, flags).
    """
    rows = np.ascontiguousarray(rows_bf16_bits)
    assert rows.dtype == np.uint16 and rows.ndim == 2
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, K = w.shape
    inv = np.ascontiguousarray(inv_permuted_idx, dtype=np.int32).reshape(-1)
    assert inv.shape[0] == T * K
    H = rows.shape[1]
    out = np.zeros((T, H), np.uint16)
    flags = lib.oracle_unpermute(_ptr(rows), rows.shape[0], _ptr(w), _ptr(inv),
                                 T, H, K, _ptr(out))
    return out, int(flags)


def _f32_to_bf16_rne(lib, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.zeros(x.shape[0], np.uint16)
    lib.oracle_f32_to_bf16_rne(_ptr(x), x.shape[0], _ptr(out))
    return out
