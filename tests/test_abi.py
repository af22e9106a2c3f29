"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every function
that include/dfs.h declares (no compute calls: this runs on the CPU-only host)."""
import ctypes
import os
import re

import pytest

from draft_speculative_decoding_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dfs.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dfs_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("dfs_lmhead_topk", "dfs_pair_score", "dfs_path_select", "dfs_verify",
              "dfs_select_verify", "dfs_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    assert set(_declared_functions()) == set(binding.SIGNATURES)


def test_host_only_calls(lib):
    assert lib.dfs_version() == 1
    launches = binding.dfs_launch_count()
    assert binding.status_string(binding.DFS_ERR_WORKSPACE) == "workspace too small"
    # invalid dims are rejected on the host before any device work
    assert lib.dfs_workspace_size(None) == 0
    bad = binding.make_dims(1, 4, 1000, 256, 32, 0, 0)
    bad.K = 8
    assert lib.dfs_workspace_size(ctypes.byref(bad)) == 0
    bad = binding.make_dims(1, 17, 1024, 256, 32, 0, 0)  # block longer than 16
    assert lib.dfs_path_select(ctypes.byref(bad), None, None, 0, None, None, None) == \
        binding.DFS_ERR_UNSUPPORTED
    ok = binding.make_dims(2, 4, 1024, 256, 32, 0, 0)
    assert lib.dfs_path_select(ctypes.byref(ok), None, None, 0, None, None, None) == \
        binding.DFS_ERR_INVALID
    # a misaligned pointer is an argument error
    assert lib.dfs_path_select(ctypes.byref(ok), ctypes.c_void_p(0x1004), ctypes.c_void_p(0x2000),
                               0, ctypes.c_void_p(0x3000), None, None) == binding.DFS_ERR_INVALID
    assert lib.dfs_path_select(ctypes.byref(ok), ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000),
                               7, ctypes.c_void_p(0x3000), None, None) == binding.DFS_ERR_INVALID
    # calls rejected on the host launch nothing
    assert binding.dfs_launch_count() == launches
