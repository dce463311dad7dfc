"""ctypes binding of libmoe_permute.so (include/moe_permute.h).

Argument marshalling only: every step of permute and unpermute runs in the
CUDA library.  If the library has not been built this module raises on first
use; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import DEBUG_LIB_PATH, LIB_PATH

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_WORKSPACE_TOO_SMALL = -2
MOE_ERR_UNSUPPORTED_DEVICE = -3
MOE_ERR_CUDA = -4

MOE_DTYPE_BF16 = 0
MOE_DTYPE_FP16 = 1
MOE_DTYPE_FP8_E4M3 = 2
MOE_DTYPE_FP8_E5M2 = 3
MOE_DTYPE_FP32 = 4

MOE_INDEX_INT32 = 0
MOE_INDEX_INT64 = 1

MOE_FLAG_ID_OUT_OF_RANGE = 1
MOE_FLAG_MAP_OUT_OF_RANGE = 2
MOE_FLAG_INV_OUT_OF_RANGE = 4
MOE_FLAG_BARRIER_TIMEOUT = 8
MOE_FLAG_CAPACITY_OVERFLOW = 16

MOE_MAX_TOPK = 32
MOE_MAX_LOCAL_EXPERTS = 1024
MOE_QUANT_GROUP = 128

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/moe_permute.h
SIGNATURES = {
    "moe_permute_supported": (ctypes.c_int, [ctypes.c_int]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_permute_workspace_size": (_SZ, [_I64, _I32, _I32]),
    "moe_permute_workspace_init": (ctypes.c_int, [_P, _SZ, _P]),
    "moe_permute": (ctypes.c_int, [_P, ctypes.c_int, _P, _I64, _P, ctypes.c_int, _P,
                                   _I64, _I64, _I32, _I32, _I32,
                                   _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_unpermute": (ctypes.c_int, [_P, _I64, _P, _P, _I64, _I64, _I32, _P, _P, _P]),
    "moe_read_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "moe_clear_status": (ctypes.c_int, [_P, _P]),
    "moe_permute_read_status": (ctypes.c_int, [_P, _P, ctypes.c_int, _P]),
    "moe_permute_batched": (ctypes.c_int, [_P, ctypes.c_int, _P, _I64, _P, ctypes.c_int, _P,
                                           _I64, _I64, _I32, _I32, _I32, _I64,
                                           _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_quant_fp8": (ctypes.c_int, [_P, _P, ctypes.c_int, _P, _I64, _I64, _I32, _I32,
                                             _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (ctypes.c_int, [_P, ctypes.c_int, _P, _I64, _P, ctypes.c_int, _P,
                                           _I64, _I64, _I32, _I32, _I32,
                                           _P, _P, _P, _P, _P, _P]),
}

MOE_NOALLOC_SCRATCH_BYTES = (1 << 20) + 256

# Exported by the debug build only (include/moe_permute_debug.h).
DEBUG_SIGNATURES = {
    "moe_debug_set_table_wait": (ctypes.c_int, [ctypes.c_int, ctypes.c_ulonglong]),
    "moe_debug_check_quant_division": (ctypes.c_int, [ctypes.POINTER(ctypes.c_ulonglong)]),
}
MOE_DEBUG_MAX_EXTRA_ROWS = 4
TABLE_WAIT_NS = 2_000_000_000  # the production limit of a routing-table wait

_lib = None
_debug_lib = None
_lock = threading.Lock()


class MoeError(RuntimeError):
    """A C-ABI entry point returned a negative status."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def library_path() -> str:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was never built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -c 'import __graft_entry__ as g; g.build()'` "
                        "(this package has no CPU fallback)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def debug_lib() -> ctypes.CDLL:
    """The debug build (same entry points plus the test hook); for tests."""
    global _debug_lib
    if _debug_lib is None:
        with _lock:
            if _debug_lib is None:
                if not os.path.exists(DEBUG_LIB_PATH):
                    raise RuntimeError(f"{DEBUG_LIB_PATH} is missing: build it with "
                                       "`python -c 'import __graft_entry__ as g; g.build()'`")
                handle = ctypes.CDLL(DEBUG_LIB_PATH)
                for name, (res, args) in {**SIGNATURES, **DEBUG_SIGNATURES}.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _debug_lib = handle
    return _debug_lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoeError(fn, status)
