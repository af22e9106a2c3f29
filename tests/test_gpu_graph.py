"""The fused call inside a CUDA graph (the pages' serving setups decode under CUDA graphs):
dfs_select_verify allocates, frees and synchronises nothing and makes no runtime call but
its launches once warmed up, so a capture records it; replays must reproduce eager results
bit for bit."""
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl
from parity import dims_for

pytestmark = pytest.mark.gpu

CASES = [
    wl.TINY.with_(name="graph_small", dtype="bf16", B=4, L=8, V=5000, d=256, r=64, seed=51),
    wl.TINY.with_(name="graph_pairs", dtype="bf16", B=24, L=8, V=5000, d=256, r=256, seed=52,
                  zipf=True),
]
CALLS = [(binding.DFS_PATH_GREEDY, 0.0, 3), (binding.DFS_PATH_VITERBI, 0.8, 4),
         (binding.DFS_PATH_SAMPLE, 0.8, 5)]


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def _outputs(spec):
    P = spec.L - 1
    return (torch.zeros(spec.B, P, dtype=torch.int32, device="cuda"),
            torch.zeros(spec.B, spec.L, dtype=torch.int32, device="cuda"),
            torch.zeros(spec.B, dtype=torch.int32, device="cuda"))


def _call(data, dims, ws, mode, T, seed, outs):
    binding.dfs_select_verify(dims, data["h"], data["W"], data["Wg"], data["A"], data["Bt"],
                              data["x0"], data["Z"], mode, T, seed, ws, outputs=outs)


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_fused_call_replays_from_a_cuda_graph(lib, spec):
    data = wl.generate(spec, "cuda")
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    eager = []
    for mode, T, seed in CALLS:
        outs = _outputs(spec)
        _call(data, dims, ws, mode, T, seed, outs)
        eager.append([o.clone() for o in outs])
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK

    graph_outs = [_outputs(spec) for _ in CALLS]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up off the default stream, as capture requires
        for (mode, T, seed), outs in zip(CALLS, graph_outs):
            _call(data, dims, ws, mode, T, seed, outs)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (mode, T, seed), outs in zip(CALLS, graph_outs):
            _call(data, dims, ws, mode, T, seed, outs)
    for outs in graph_outs:
        for o in outs:
            o.fill_(-7)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for ref, outs in zip(eager, graph_outs):
            for a, b in zip(ref, outs):
                assert torch.equal(a, b)
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
