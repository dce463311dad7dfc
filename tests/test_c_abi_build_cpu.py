"""The boundary as C: the public headers compile as strict C99 and C++17, and
a plain C program using the ABI (no Python, no torch) builds and links."""
import os
import subprocess

import pytest

from c_abi_build import ROOT, build_consumer

HEADERS = ["moe_permute.h", "moe_permute_debug.h"]


@pytest.mark.parametrize("header", HEADERS)
@pytest.mark.parametrize("lang,std,compiler", [("c", "-std=c99", "gcc"),
                                               ("c++", "-std=c++17", "g++")])
def test_header_compiles_strictly(header, lang, std, compiler):
    subprocess.check_call([compiler, std, "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-fsyntax-only", "-x", lang,
                           os.path.join(ROOT, "include", header)])


def test_c_consumer_builds(tmp_path):
    exe = build_consumer(str(tmp_path))
    assert os.access(exe, os.X_OK)
