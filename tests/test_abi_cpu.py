"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every
entry point include/pmha.h declares; host-side argument checks that return
before any device work behave as documented. No kernel runs here."""
import ctypes
import os
import re

import pytest

from graph_sparse_head_gb300 import _lib
from graph_sparse_head_gb300 import build as pmha_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pmha.h")


@pytest.fixture(scope="module")
def lib():
    pmha_build.build()
    return _lib.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pmha_[a-z_]+)\s*\(", text)))


def test_header_declares_the_calls_of_the_boundary():
    names = declared_functions()
    for n in ("pmha_build_csr", "pmha_forward", "pmha_edge_weights", "pmha_graph_destroy",
              "pmha_forward_workspace_size", "pmha_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature in the binding"
    assert set(_lib.SIGNATURES) == set(names)


def test_library_is_built_for_sm_103a_only():
    assert any("arch=compute_103a,code=sm_103a" in f for f in pmha_build.ARCH)
    assert len([f for f in pmha_build.ARCH if f.startswith("arch=")]) == 1


def test_host_checks_before_device_work(lib):
    out = ctypes.c_void_p(123)
    # nnz < 1 -> PMHA_ERR_EMPTY, out set to NULL
    st = lib.pmha_build_csr(None, None, 0, 4, 4, 0, None, ctypes.byref(out))
    assert st == 4 and out.value is None
    assert b"empty" in lib.pmha_last_error()
    # NULL out
    assert lib.pmha_build_csr(None, None, 1, 4, 4, 0, None, None) == 1
    # self-loops need L == S
    st = lib.pmha_build_csr(ctypes.c_void_p(64), ctypes.c_void_p(64), 3, 4, 5, 1, None, ctypes.byref(out))
    assert st == 1 and b"query_features == key_features" in lib.pmha_last_error()
    # non-positive sizes
    assert lib.pmha_build_csr(ctypes.c_void_p(64), ctypes.c_void_p(64), 3, 0, 5, 0, None, ctypes.byref(out)) == 1
    # misaligned index pointers
    assert lib.pmha_build_csr(ctypes.c_void_p(65), ctypes.c_void_p(64), 3, 4, 4, 0, None, ctypes.byref(out)) == 1
    # NULL graph / params
    assert lib.pmha_forward(None, None, None, None, None, None, 1, None, 0, None, None, 0, None) == 1
    assert lib.pmha_edge_weights(None, None, None, None, None, 1, 1, None, None, 0, None) == 1
    assert lib.pmha_forward_workspace_size(None, None, 1, 0) == 0
    assert lib.pmha_graph_info(None, None, None, None, None) == 1
    assert lib.pmha_graph_split_info(None, None, None, None) == 1
    lib.pmha_graph_destroy(None)
    assert lib.pmha_profile_enable(0) == 0
    assert lib.pmha_launch_count() >= 0


def test_status_names_cover_the_header():
    with open(HEADER) as f:
        text = f.read()
    for name in re.findall(r"\b(PMHA_(?:OK|ERR_[A-Z_]+))\s*=", text):
        assert name in _lib.STATUS_NAMES.values(), name
