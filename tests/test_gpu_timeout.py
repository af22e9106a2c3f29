"""Failure detection on the GPU without a fault: every wait in the LM-head kernels is
bounded, and a wait that runs out sets the workspace's error word, stops every role of the
CTA and returns, so the host reads DFS_ERR_TIMEOUT and the context stays usable.

The test keeps the MMA issuer idle (a test hook read by the library on each call) with a
short wait limit: the TMA producers fill their rings (those copies land within microseconds)
and then wait for stages that are never released, the epilogue waits for accumulators that
never fill; both give up after the limit. A normal call follows on the same context and must
be correct."""
import numpy as np
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl
from parity import compare_topk, dims_for, np_inputs, to_cpu

pytestmark = pytest.mark.gpu

CASES = [
    # <= 128 rows: k_lmhead_tc (clusters sharing the hidden rows)
    wl.TINY.with_(name="timeout_small", dtype="bf16", B=4, L=8, V=4096, d=256, r=64, seed=41),
    # 129..256 rows: k_lmhead_pair (CTA pairs, pair MMAs)
    wl.TINY.with_(name="timeout_pairs", dtype="bf16", B=24, L=8, V=4096, d=256, r=64, seed=42),
]


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def _oracle_topk(orc, npd, spec):
    rows = np.array([b * spec.L + t for b in range(spec.B) for t in range(1, spec.L)])
    u = orc.logits(npd["h"], npd["W"], rows)
    ids, U, gap = orc.topk(u, 16)
    P = spec.L - 1
    return ids.reshape(spec.B, P, 16), U.reshape(spec.B, P, 16), gap.reshape(spec.B, P)


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_wait_runs_out_reports_timeout_and_context_survives(lib, orc, spec, monkeypatch):
    data = wl.generate(spec, "cuda")
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK

    monkeypatch.setenv("DFS_DEBUG_WAIT_LIMIT_NS", "2000000")  # 2 ms
    monkeypatch.setenv("DFS_DEBUG_STALL_MMA", "1")
    binding.dfs_lmhead_topk(dims, data["h"], data["W"], ws)
    torch.cuda.synchronize()  # the kernel returned: no hang
    assert binding.dfs_get_device_error(ws) == binding.DFS_ERR_TIMEOUT
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK  # read-and-clear

    # the fused call reports the LM head's timeout too (the tail runs on and returns)
    binding.dfs_select_verify(dims, data["h"], data["W"], data["Wg"], data["A"], data["Bt"],
                              data["x0"], data["Z"], binding.DFS_PATH_GREEDY, 0.0, 1, ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_ERR_TIMEOUT

    monkeypatch.delenv("DFS_DEBUG_STALL_MMA")
    monkeypatch.delenv("DFS_DEBUG_WAIT_LIMIT_NS")
    ids, U = binding.dfs_lmhead_topk(dims, data["h"], data["W"], ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    o_ids, o_U, o_gap = _oracle_topk(orc, np_inputs(data), spec)
    n, near, diverged = compare_topk(to_cpu(ids), to_cpu(U), o_ids, o_U, o_gap)
    assert diverged <= max(1, n // 50)
