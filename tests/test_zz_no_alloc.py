"""dfs_verify_noalloc: verification for callers that cannot allocate device memory (a step
handed only its inputs and outputs, a pool owned by another component, a thread that must not
enter the CUDA allocator). It must give exactly what dfs_verify gives with a workspace, on
consecutive calls that reuse its built-in scratch.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process (it builds and loads the
library itself)."""
import ctypes

import numpy as np
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import build as dfs_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    dfs_build.build()
    return binding.load()


def _case(seed, B, L, V, zdtype):
    rng = np.random.default_rng(seed)
    Z = torch.from_numpy((rng.standard_normal((B, L, V)) * 3).astype(np.float32)).cuda()
    if zdtype == binding.DFS_BF16:
        Z = Z.to(torch.bfloat16)
    y = Z.float().argmax(-1).cpu().numpy()
    path = y[:, :L - 1].copy()
    flip = rng.random(path.shape) > 0.8
    path[flip] = (path[flip] + 1 + rng.integers(0, 50, flip.sum())) % V
    return Z, torch.from_numpy(path.astype(np.int32)).cuda()


@pytest.mark.parametrize("T", [0.0, 0.8])
@pytest.mark.parametrize("zdtype", [binding.DFS_BF16, binding.DFS_FP32])
def test_noalloc_matches_workspace_verify_twice(lib, T, zdtype):
    B, L, V = 12, 8, 3 * 8192 + 40
    dims = binding.make_dims(B, L, V, 64, 8, zdtype, zdtype)
    ws = binding.alloc_workspace(dims)
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        Z, path = _case(seed + int(T * 10) + zdtype, B, L, V, zdtype)
        ref_out, ref_acc = binding.dfs_verify(dims, path, Z, T, 900 + call, ws)
        out, acc = binding.dfs_verify_noalloc(dims, path, Z, T, 900 + call)
        torch.cuda.synchronize()
        assert torch.equal(acc, ref_acc), f"call {call}: accept lengths differ"
        assert torch.equal(out, ref_out), f"call {call}: emitted tokens differ"


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    """22 requests of 16 positions over the largest vocabulary (4194304 tokens, 1024 chunks)
    need more than the built-in 4 MiB of row statistics: the call returns DFS_ERR_WORKSPACE.
    Every buffer is real and as large as the shape says (the target logits take 2.95 GB), so
    nothing the call could launch would read outside them."""
    B, L, V = 22, 16, 4194304
    dims = binding.make_dims(B, L, V, 64, 8, binding.DFS_BF16, binding.DFS_BF16)
    Z = torch.empty(B, L, V, dtype=torch.bfloat16, device="cuda")
    path = torch.zeros(B, L - 1, dtype=torch.int32, device="cuda")
    out = torch.empty(B, L, dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    before = binding.dfs_launch_count()
    rc = lib.dfs_verify_noalloc(ctypes.byref(dims), binding._ptr(path), binding._ptr(Z), 0.0, 0,
                                binding._ptr(out), binding._ptr(acc), None)
    assert rc == binding.DFS_ERR_WORKSPACE
    assert binding.dfs_launch_count() == before  # rejected before anything was enqueued
    del Z


@pytest.mark.parametrize("T", [0.0, 0.8])
def test_noalloc_more_rows_than_one_grid_dimension(lib, T):
    """70000 target rows (more than a grid's second dimension holds) fit the scratch at a
    4096-token vocabulary; two calls in a row agree with dfs_verify."""
    B, L, V = 4375, 16, 4096
    dims = binding.make_dims(B, L, V, 64, 8, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    gen = torch.Generator("cuda").manual_seed(17)
    for call in range(2):
        Z = (torch.randn(B, L, V, device="cuda", generator=gen) * 3).to(torch.bfloat16)
        path = Z.float().argmax(-1)[:, :L - 1].to(torch.int32).contiguous()
        path[::3, 2] = (path[::3, 2] + 1) % V
        ref_out, ref_acc = binding.dfs_verify(dims, path, Z, T, 40 + call, ws)
        out, acc = binding.dfs_verify_noalloc(dims, path, Z, T, 40 + call)
        torch.cuda.synchronize()
        assert torch.equal(acc, ref_acc) and torch.equal(out, ref_out), f"call {call}"
