"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every function
that include/dfs.h declares (no compute calls: this runs on the CPU-only host)."""
import ctypes
import os
import re

import pytest
import torch

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


def test_host_limits_of_the_convolution_and_the_hand_off(lib):
    launches = binding.dfs_launch_count()
    ws = lib.dfs_conv2tap_workspace_size
    assert ws(32, 8, 5120) > 256                  # error word + partial sums
    assert ws(2, 4, 96) == 0                      # d not a multiple of 64
    assert ws(1, 1, 32) == 0                      # d below 64
    assert ws(1 << 12, 1 << 11, 64) == 0          # more than 2^22 rows
    assert ws(1 << 11, 1 << 11, 64) > 0
    P = ctypes.c_void_p
    assert lib.dfs_conv2tap(2, 4, 96, P(0x1000), P(0x2000), P(0x3000), P(0x4000), P(0x5000),
                            1 << 20, None) == binding.DFS_ERR_UNSUPPORTED
    # out overlapping x is an argument error, found before anything is enqueued
    assert lib.dfs_conv2tap(2, 4, 128, P(0x10000), P(0x2000), P(0x3000), P(0x10100), P(0x5000),
                            1 << 20, None) == binding.DFS_ERR_INVALID
    assert lib.dfs_next_tokens(0, 8, P(0x1000), P(0x2000), P(0x3000), None) == binding.DFS_ERR_INVALID
    assert lib.dfs_next_tokens(4, 17, P(0x1000), P(0x2000), P(0x3000), None) == binding.DFS_ERR_INVALID
    big = binding.make_dims(65536, 2, 1024, 256, 32, 0, 0)  # more requests than the grid holds
    assert lib.dfs_path_select(ctypes.byref(big), None, None, 0, None, None, None) == \
        binding.DFS_ERR_UNSUPPORTED
    assert binding.dfs_launch_count() == launches


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only check; the GPU test covers it there")
def test_noalloc_host_checks(lib):
    """dfs_verify_noalloc rejects on the host, before any device call: a shape whose row
    statistics exceed its built-in scratch (DFS_ERR_WORKSPACE), the shapes dfs_verify
    rejects (the same checks), and a negative temperature."""
    P = ctypes.c_void_p
    launches = binding.dfs_launch_count()
    args = (P(0x1000), P(0x2000), 0.0, 0, P(0x3000), P(0x4000), None)
    big = binding.make_dims(22, 16, 4194304, 64, 8, 0, 0)
    assert lib.dfs_verify_noalloc(ctypes.byref(big), *args) == binding.DFS_ERR_WORKSPACE
    for B, L, V, K in ((65536, 2, 1024, 16), (2, 17, 1024, 16), (2, 8, 1020, 16), (2, 8, 1024, 8)):
        dims = binding.make_dims(B, L, V, 64, 8, 0, 0)
        dims.K = K
        assert lib.dfs_verify_noalloc(ctypes.byref(dims), *args) == binding.DFS_ERR_UNSUPPORTED
        assert lib.dfs_verify(ctypes.byref(dims), P(0x1000), P(0x2000), 0.0, 0, P(0x3000),
                              P(0x4000), P(0x5000), 1 << 30, None) == binding.DFS_ERR_UNSUPPORTED
    ok = binding.make_dims(2, 8, 1024, 64, 8, 0, 0)
    assert lib.dfs_verify_noalloc(ctypes.byref(ok), P(0x1000), P(0x2000), -1.0, 0, P(0x3000),
                                  P(0x4000), None) == binding.DFS_ERR_INVALID
    assert binding.dfs_launch_count() == launches
