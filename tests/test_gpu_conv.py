"""GPU parity of the two-tap dynamic depthwise convolution (include/dfs.h: dfs_conv2tap)
against the oracle's fp64 definition ("DFlash 2: Keep Drafting Parallel", §"A lightweight
local convolution"). The kernel's output is bf16 rounded once from fp32 arithmetic, so the
bar is: every element within one bf16 ulp of the exact value, and at least 99.9 % equal to
the exact value rounded to bf16 (the rest sit next to a rounding midpoint)."""
import numpy as np
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def _orc_inputs(data, blocks=None):
    x = data["x"] if blocks is None else data["x"][blocks]
    return wl.to_numpy_bits(x), data["base"].cpu().numpy(), wl.to_numpy_bits(data["Wc"])


def _compare(got, exact):
    got = got.float().cpu().numpy().astype(np.float64)
    rounded = torch.from_numpy(exact).float().to(torch.bfloat16).float().numpy().astype(np.float64)
    mag = np.maximum(np.abs(exact), 1e-30)
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    assert np.all(np.abs(got - exact) <= ulp + 1e-6), float(np.max(np.abs(got - exact) / ulp))
    assert np.mean(got == rounded) >= 0.999


SHAPES = [
    wl.CONV_SMALL,                                                    # 15 rows, one N tile
    wl.ConvSpec("conv_ragged", B=24, L=8, d=1024, seed=21),           # 2 row tiles, N 80 + 48
    wl.ConvSpec("conv_L1_d64", B=5, L=1, d=64, seed=22),              # no predecessor at all
    wl.ConvSpec("conv_long", B=4, L=16, d=2048, seed=23),
    wl.ConvSpec("conv_rows_129", B=43, L=3, d=576, seed=24),          # 129 rows: a 1-row tile
]


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
def test_conv2tap_matches_oracle(lib, orc, spec):
    data = wl.conv_inputs(spec, "cuda")
    ws = binding.alloc_conv_workspace(spec.B, spec.L, spec.d)
    out = binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    _compare(out, orc.conv2tap(*_orc_inputs(data)))


def test_conv2tap_full_size_sampled_blocks(lib, orc):
    spec = wl.CONV_THROUGHPUT
    data = wl.conv_inputs(spec, "cuda")
    ws = binding.alloc_conv_workspace(spec.B, spec.L, spec.d)
    out = binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    blocks = [0, 17, 31]  # blocks are independent: the oracle takes just these
    _compare(out[blocks], orc.conv2tap(*_orc_inputs(data, blocks)))


def test_conv2tap_is_deterministic_and_leaves_inputs(lib):
    spec = wl.ConvSpec("conv_det", B=16, L=8, d=2048, seed=25)
    data = wl.conv_inputs(spec, "cuda")
    x0 = data["x"].clone()
    ws = binding.alloc_conv_workspace(spec.B, spec.L, spec.d)
    a = binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws)
    b = binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(data["x"], x0)


def test_conv2tap_rejects_bad_arguments_on_the_host(lib):
    spec = wl.ConvSpec("conv_bad", B=2, L=4, d=128, seed=26)
    data = wl.conv_inputs(spec, "cuda")
    ws = binding.alloc_conv_workspace(spec.B, spec.L, spec.d)
    with pytest.raises(binding.DfsError) as e:  # in place: out overlaps x
        binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws, out=data["x"])
    assert e.value.status == binding.DFS_ERR_INVALID
    with pytest.raises(binding.DfsError) as e:  # workspace too small
        binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws[:256])
    assert e.value.status == binding.DFS_ERR_WORKSPACE
    x96 = torch.zeros(2, 4, 96, dtype=torch.bfloat16, device="cuda")  # d not a multiple of 64
    with pytest.raises(binding.DfsError) as e:
        binding.dfs_conv2tap(x96, torch.zeros(2, 96, device="cuda"),
                             torch.zeros(12, 96, dtype=torch.bfloat16, device="cuda"), ws)
    assert e.value.status == binding.DFS_ERR_UNSUPPORTED
    assert lib.dfs_conv2tap_workspace_size(2, 4, 96) == 0


def test_conv2tap_replays_from_a_cuda_graph(lib):
    spec = wl.ConvSpec("conv_graph", B=8, L=8, d=1024, seed=27)
    data = wl.conv_inputs(spec, "cuda")
    ws = binding.alloc_conv_workspace(spec.B, spec.L, spec.d)
    eager = binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws).clone()
    out = torch.zeros_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws, out=out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.dfs_conv2tap(data["x"], data["base"], data["Wc"], ws, out=out)
    out.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
