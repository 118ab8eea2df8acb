"""libasp.so loads and exports every function include/asp.h declares (no GPU needed)."""
import os
import re

import pytest

from adaptive_sparse_paged_gb300 import binding as B
from adaptive_sparse_paged_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(asp_[a-z_0-9]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        try:
            build_mod.build()
        except RuntimeError as e:  # no nvcc on this machine
            pytest.skip(str(e))
    return B.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names, "no declarations found"
    assert names == set(B.EXPORTED), names ^ set(B.EXPORTED)
    for n in names:
        assert hasattr(lib, n), f"{n} missing from libasp.so"


def test_abi_version(lib):
    src = open(os.path.join(ROOT, "include", "asp.h")).read()
    want = int(re.search(r"#define ASP_ABI_VERSION (\d+)", src).group(1))
    assert B.asp_abi_version() == want


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5):
        assert lib.asp_status_string(st).decode().startswith("ASP_")
