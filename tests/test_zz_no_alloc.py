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
    dims = binding.make_dims(4096, 16, 151936, 64, 8, binding.DFS_BF16, binding.DFS_BF16)
    rc = lib.dfs_verify_noalloc(ctypes.byref(dims), ctypes.c_void_p(0x1000),
                                ctypes.c_void_p(0x2000), 0.0, 0, ctypes.c_void_p(0x3000),
                                ctypes.c_void_p(0x4000), None)
    assert rc == binding.DFS_ERR_WORKSPACE
