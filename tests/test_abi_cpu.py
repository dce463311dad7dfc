"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and its host-only entry points (workspace sizing, status
text, argument checks that run before any device work) behave as declared."""
import ctypes
import glob
import os
import re

import pytest

from moe_token_permute_gb300 import _binding as b
from moe_token_permute_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return b.lib()


DEBUG_HEADER = "moe_permute_debug.h"  # exported by the debug build only


def declared_symbols(debug=False):
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        if (os.path.basename(h) == DEBUG_HEADER) != debug:
            continue
        with open(h) as f:
            text = f.read()
        names |= set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text))
    return names


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ("moe_permute_workspace_size", "moe_permute", "moe_unpermute",
              "moe_permute_workspace_init", "moe_permute_supported"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
        assert n in b.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_debug_hook_only_in_debug_build(lib):
    debug_names = declared_symbols(debug=True)
    assert debug_names == {"moe_debug_set_table_wait", "moe_debug_check_quant_division"}
    for n in debug_names:
        assert not hasattr(lib, n), f"{n} leaked into the production library"
    dlib = b.debug_lib()
    for n in declared_symbols() | debug_names:
        assert hasattr(dlib, n), f"{n} missing from the debug library"
        assert n in b.SIGNATURES or n in b.DEBUG_SIGNATURES


@pytest.mark.parametrize("args", [(-1, 1000), (b.MOE_DEBUG_MAX_EXTRA_ROWS + 1, 1000), (1, 0)])
def test_debug_hook_rejects_bad_arguments_on_host(lib, args):
    assert b.debug_lib().moe_debug_set_table_wait(*args) == b.MOE_ERR_INVALID_ARG


def test_division_check_rejects_null_on_host(lib):
    assert b.debug_lib().moe_debug_check_quant_division(None) == b.MOE_ERR_INVALID_ARG


def test_library_built_for_sm103a_only():
    src = open(cuda_build.__file__).read()
    assert "arch=compute_103a,code=sm_103a" in src


def test_workspace_size(lib):
    ws = lib.moe_permute_workspace_size
    assert ws(0, 1, 1) == 256 + 256  # header + one (padded) histogram row
    a = ws(4096, 2, 8)
    c = ws(32768, 8, 256)
    assert a % 256 == 0 and c % 256 == 0
    # per-block histogram table: one int per (expert, block), up to 1024 blocks
    assert c == 256 + 256 * 1024 * 4
    assert ws(100, 8, 256) <= c  # monotone in tokens
    assert ws(-1, 2, 8) == 0
    assert ws(16, 0, 8) == 0
    assert ws(16, 33, 8) == 0
    assert ws(16, 2, 0) == 0
    assert ws(2**31, 2, 8) == 0  # T*K beyond int32


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"ok"
    assert b"workspace" in lib.moe_status_string(-2)
    assert lib.moe_status_string(12345) == b"unknown status"


def _permute_args(**over):
    # a structurally valid call with fake (never dereferenced) device pointers
    args = dict(hidden=0x1000, dt=b.MOE_DTYPE_BF16, scales=None, scale_cols=0,
                ids=0x2000, idt=b.MOE_INDEX_INT32, emap=None, T=4, H=8, K=2, E=4, EL=4,
                out=0x3000, out_scales=None, offsets=0x4000, pidx=0x5000, inv=0x6000,
                ws=0x10000, ws_bytes=1 << 20, stream=None)
    args.update(over)
    return list(args.values())


@pytest.mark.parametrize("over", [
    dict(K=0), dict(K=33), dict(E=0), dict(EL=5), dict(EL=2),  # EL != E without a map
    dict(EL=1025, E=2000, emap=0x7000), dict(T=-1), dict(H=0), dict(dt=9), dict(idt=3),
    dict(ids=None), dict(ids=0x2002), dict(offsets=0x4004), dict(pidx=None), dict(inv=0x6002),
    dict(hidden=None), dict(scales=0x8000), dict(scale_cols=3), dict(ws=None),
    dict(ws=0x10010), dict(T=2**30, K=4),
])
def test_permute_rejects_bad_arguments_on_host(lib, over):
    assert lib.moe_permute(*_permute_args(**over)) == b.MOE_ERR_INVALID_ARG


def test_permute_workspace_too_small(lib):
    assert lib.moe_permute(*_permute_args(T=100000, ws_bytes=512)) == b.MOE_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("args", [
    (0x1000, 4, 0x2000, 0x3000, 4, 8, 0, 0x4000, None, None),   # K = 0
    (0x1000, 4, 0x2000, 0x3000, 4, 8, 40, 0x4000, None, None),  # K > 32
    (0x1000, 4, 0x2000, 0x3000, 4, 0, 2, 0x4000, None, None),   # H = 0
    (0x1000, 4, None, 0x3000, 4, 8, 2, 0x4000, None, None),     # weights NULL
    (0x1000, 4, 0x2000, 0x3000, 4, 8, 2, 0x4001, None, None),   # out misaligned
    (0x1000, 4, 0x2000, 0x3000, 4, 8, 2, 0x4000, 0x10010, None),  # ws misaligned
])
def test_unpermute_rejects_bad_arguments_on_host(lib, args):
    assert lib.moe_unpermute(*args) == b.MOE_ERR_INVALID_ARG


def test_unpermute_empty_batch_is_a_no_op(lib):
    assert lib.moe_unpermute(None, 0, None, None, 0, 8, 2, None, None, None) == b.MOE_OK


def test_status_calls_reject_bad_workspace(lib):
    v = ctypes.c_uint32(0)
    assert lib.moe_read_status(None, ctypes.byref(v), None) == b.MOE_ERR_INVALID_ARG
    assert lib.moe_clear_status(0x10010, None) == b.MOE_ERR_INVALID_ARG
    assert lib.moe_permute_workspace_init(0x10000, 16, None) == b.MOE_ERR_INVALID_ARG
    # the asynchronous read: NULL or misaligned workspace, NULL or misaligned dst
    assert lib.moe_permute_read_status(None, 0x2000, 0, None) == b.MOE_ERR_INVALID_ARG
    assert lib.moe_permute_read_status(0x10010, 0x2000, 0, None) == b.MOE_ERR_INVALID_ARG
    assert lib.moe_permute_read_status(0x10000, None, 1, None) == b.MOE_ERR_INVALID_ARG
    assert lib.moe_permute_read_status(0x10000, 0x2002, 1, None) == b.MOE_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        b.lib()


def _quant_args(**over):
    # moe_permute_quant_fp8 with fake (never dereferenced) device pointers
    args = dict(hidden=0x1000, ids=0x2000, idt=b.MOE_INDEX_INT32, emap=None, T=4, H=256, K=2,
                E=4, EL=4, codes=0x3000, scales=0x8000, offsets=0x4000, pidx=0x5000,
                inv=0x6000, ws=0x10000, ws_bytes=1 << 20, stream=None)
    args.update(over)
    return list(args.values())


@pytest.mark.parametrize("over", [
    dict(H=100), dict(H=64), dict(H=0), dict(K=0), dict(K=33), dict(E=0), dict(EL=5),
    dict(EL=2),  # EL != E without a map
    dict(T=-1), dict(idt=3), dict(offsets=None), dict(offsets=0x4004), dict(ids=None),
    dict(ids=0x2002), dict(pidx=None), dict(inv=0x6002), dict(hidden=None),
    dict(hidden=0x1008),  # bf16 rows are read in 16-byte vectors
    dict(codes=None), dict(codes=0x3004), dict(scales=None), dict(scales=0x8002),
    dict(ws=None), dict(ws=0x10010), dict(T=2**30, K=4),
])
def test_quant_permute_rejects_bad_arguments_on_host(lib, over):
    assert lib.moe_permute_quant_fp8(*_quant_args(**over)) == b.MOE_ERR_INVALID_ARG


def test_quant_permute_workspace_too_small(lib):
    assert (lib.moe_permute_quant_fp8(*_quant_args(T=100000, ws_bytes=512))
            == b.MOE_ERR_WORKSPACE_TOO_SMALL)


def _batched_args(**over):
    # moe_permute_batched with fake (never dereferenced) device pointers
    args = dict(hidden=0x1000, dt=b.MOE_DTYPE_BF16, scales=None, scale_cols=0, ids=0x2000,
                idt=b.MOE_INDEX_INT32, emap=None, T=4, H=8, K=2, E=4, EL=4, M=8, out=0x3000,
                out_scales=None, counts=0x4000, inv=0x6000, ws=0x10000, ws_bytes=1 << 20,
                stream=None)
    args.update(over)
    return list(args.values())


@pytest.mark.parametrize("over", [
    dict(dt=9), dict(M=0), dict(M=-3), dict(M=2**31 // 4 + 1),  # E_L * M beyond int32
    dict(K=0), dict(K=33), dict(E=0), dict(EL=2), dict(T=-1), dict(H=0), dict(idt=3),
    dict(counts=None), dict(counts=0x4002), dict(ids=None), dict(inv=None), dict(inv=0x6002),
    dict(hidden=None),  # rows asked for without a source
    dict(scales=0x8000),  # source scales without output scales
    dict(scales=0x8000, out_scales=0x9000, scale_cols=0),
    dict(scale_cols=2),  # a scale width without scales
    dict(ws=None), dict(ws=0x10010),
])
def test_batched_permute_rejects_bad_arguments_on_host(lib, over):
    assert lib.moe_permute_batched(*_batched_args(**over)) == b.MOE_ERR_INVALID_ARG


def test_batched_permute_workspace_too_small(lib):
    assert (lib.moe_permute_batched(*_batched_args(T=100000, ws_bytes=512))
            == b.MOE_ERR_WORKSPACE_TOO_SMALL)


def test_noalloc_rejects_problems_beyond_its_scratch_on_host(lib):
    # 512 experts: the histogram table alone outgrows the library's fixed scratch,
    # which the call reports before it touches a device
    assert lib.moe_permute_workspace_size(4096, 2, 512) > b.MOE_NOALLOC_SCRATCH_BYTES
    args = list(dict(hidden=0x1000, dt=b.MOE_DTYPE_BF16, scales=None, scale_cols=0, ids=0x2000,
                     idt=b.MOE_INDEX_INT32, emap=None, T=4096, H=8, K=2, E=512, EL=512,
                     out=0x3000, out_scales=None, offsets=0x4000, pidx=0x5000, inv=0x6000,
                     stream=None).values())
    assert lib.moe_permute_noalloc(*args) == b.MOE_ERR_WORKSPACE_TOO_SMALL


def _noalloc_args(**over):
    args = dict(hidden=0x1000, dt=b.MOE_DTYPE_BF16, scales=None, scale_cols=0, ids=0x2000,
                idt=b.MOE_INDEX_INT32, emap=None, T=4096, H=8, K=2, E=512, EL=512,
                out=0x3000, out_scales=None, offsets=0x4000, pidx=0x5000, inv=0x6000,
                stream=None)
    args.update(over)
    return list(args.values())


@pytest.mark.parametrize("over", [dict(K=0), dict(ids=None), dict(EL=5), dict(offsets=0x4004),
                                  dict(dt=9), dict(scale_cols=3)])
def test_noalloc_checks_arguments_before_its_scratch_size(lib, over):
    # invalid arguments are reported as such, even for a problem the static
    # scratch could not hold
    assert lib.moe_permute_noalloc(*_noalloc_args(**over)) == b.MOE_ERR_INVALID_ARG


def test_noalloc_empty_batch_fits_whatever_the_expert_count(lib):
    # T = 0 needs no table: not MOE_ERR_WORKSPACE_TOO_SMALL even with 1024 experts
    # (without a GPU the call then stops at the device lookup)
    rc = lib.moe_permute_noalloc(*_noalloc_args(T=0, E=1024, EL=1024, hidden=None, out=None,
                                                ids=None, pidx=None, inv=None))
    assert rc in (b.MOE_OK, b.MOE_ERR_CUDA)
