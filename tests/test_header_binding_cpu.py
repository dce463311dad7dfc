"""The Python binding mirrors include/moe_permute.h by hand (status codes,
dtype and index enums, flag bits, limits, and every entry point's argument
list).  These tests hold the two together: a C program compiled against the
header prints every constant, and each prototype's parameter count must match
its ctypes signature."""
import os
import re
import shutil
import subprocess

import pytest

from moe_token_permute_gb300 import _binding as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

CONSTANTS = [
    "MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_WORKSPACE_TOO_SMALL", "MOE_ERR_UNSUPPORTED_DEVICE",
    "MOE_ERR_CUDA", "MOE_DTYPE_BF16", "MOE_DTYPE_FP16", "MOE_DTYPE_FP8_E4M3",
    "MOE_DTYPE_FP8_E5M2", "MOE_DTYPE_FP32", "MOE_INDEX_INT32", "MOE_INDEX_INT64",
    "MOE_FLAG_ID_OUT_OF_RANGE", "MOE_FLAG_MAP_OUT_OF_RANGE", "MOE_FLAG_INV_OUT_OF_RANGE",
    "MOE_FLAG_BARRIER_TIMEOUT", "MOE_FLAG_CAPACITY_OVERFLOW", "MOE_MAX_TOPK",
    "MOE_MAX_LOCAL_EXPERTS", "MOE_QUANT_GROUP", "MOE_NOALLOC_SCRATCH_BYTES",
    "MOE_DEBUG_MAX_EXTRA_ROWS",
]


@pytest.fixture(scope="module")
def header_values(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    d = tmp_path_factory.mktemp("hdr")
    src = d / "consts.c"
    body = "\n".join(f'    printf("{n} %lld\\n", (long long)({n}));' for n in CONSTANTS)
    src.write_text('#include <stdio.h>\n#include "moe_permute.h"\n#include "moe_permute_debug.h"\n'
                   f"int main(void) {{\n{body}\n    return 0;\n}}\n")
    exe = d / "consts"
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", INCLUDE, "-o", str(exe), str(src)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (ln.split() for ln in out.splitlines())}


@pytest.mark.parametrize("name", CONSTANTS)
def test_binding_constant_matches_header(header_values, name):
    assert getattr(b, name) == header_values[name]


def prototypes():
    """name -> parameter count of every MOE_API function in include/*.h."""
    found = {}
    for h in sorted(os.listdir(INCLUDE)):
        text = open(os.path.join(INCLUDE, h)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        for m in re.finditer(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(([^)]*)\)\s*;", text):
            params = m.group(2).strip()
            found[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return found


def test_every_prototype_has_a_signature_of_the_same_arity():
    protos = prototypes()
    assert "moe_permute" in protos and "moe_debug_set_table_wait" in protos
    sigs = {**b.SIGNATURES, **b.DEBUG_SIGNATURES}
    assert set(protos) == set(sigs)
    for name, n in protos.items():
        assert len(sigs[name][1]) == n, name
