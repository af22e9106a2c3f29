"""GPU parity of the E4M3 LM head (include/dfs.h: dfs_quantize_rows_e4m3,
dfs_lmhead_topk_e4m3, dfs_select_verify_e4m3) against the oracle's E4M3 definitions: the
quantised rows and scales bit for bit, then the top-16 and the whole step as for bf16."""
import numpy as np
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl
from parity import compare_topk, dims_for, np_inputs, oracle_head, oracle_step, to_cpu
from test_gpu_fused import _compare, _invariants

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def test_row_quantisation_is_bit_exact(lib, orc):
    B, L, d = 5, 8, 384
    g = torch.Generator(device="cuda").manual_seed(8)
    h = torch.randn(B, L, d, generator=g, device="cuda") * 3.0
    h[0, 1] = 0.0                                   # zero row: scale 1
    h[0, 2] = 0.0
    h[0, 2, 5] = 448.0 * 2.0 ** -3                  # the scale boundary
    h[1, 0] *= 2.0 ** -40                           # tiny row
    h[2, 3] *= 2.0 ** 20                            # large row
    h = h.to(torch.bfloat16)
    dims = binding.make_dims(B, L, 4096, d, 64, binding.DFS_BF16, binding.DFS_BF16)
    q, sc = binding.dfs_quantize_rows_e4m3(dims, h)
    torch.cuda.synchronize()
    oq, osc = orc.quantize_rows_e4m3(wl.to_numpy_bits(h), np.arange(B * L))
    assert np.array_equal(to_cpu(sc).astype(np.float64), osc)
    assert np.array_equal(to_cpu(q), oq)


SHAPES = [
    wl.TINY.with_(name="q_mt1", dtype="bf16", B=3, L=5, V=5000, d=256, r=64, seed=61,
                  lmhead="e4m3"),
    wl.TINY.with_(name="q_pairs", dtype="bf16", B=24, L=8, V=4000, d=384, r=256, seed=62,
                  zipf=True, lmhead="e4m3"),
    wl.TINY.with_(name="q_groups", dtype="bf16", B=40, L=8, V=2048, d=128, r=64, seed=63,
                  lmhead="e4m3"),
]


def _oracle_topk(orc, npd, data, spec):
    rows = np.array([b * spec.L + t for b in range(spec.B) for t in range(1, spec.L)])
    q, s = orc.quantize_rows_e4m3(npd["h"], rows)
    u = orc.logits_e4m3(q, s, to_cpu(data["Wq"]), to_cpu(data["w_scale"]))
    ids, U, gap = orc.topk(u, 16)
    P = spec.L - 1
    return ids.reshape(spec.B, P, 16), U.reshape(spec.B, P, 16), gap.reshape(spec.B, P)


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
def test_lmhead_topk_e4m3(lib, orc, spec):
    data = wl.generate(spec, "cuda")
    npd = np_inputs(data)
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    Wp = binding.dfs_pack_e4m3_head(data["Wq"])
    ids, U = binding.dfs_lmhead_topk_e4m3(dims, data["h"], Wp, data["w_scale"], ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    o_ids, o_U, o_gap = _oracle_topk(orc, npd, data, spec)
    n, near, diverged = compare_topk(to_cpu(ids), to_cpu(U), o_ids, o_U, o_gap)
    assert diverged <= max(1, n // 50), f"{diverged}/{n} rows diverged on near-ties ({near} near)"


def _run_e4m3(data, spec, mode, T, seed):
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    Wp = binding.dfs_pack_e4m3_head(data["Wq"])
    res = binding.dfs_select_verify_e4m3(dims, data["h"], Wp, data["w_scale"], data["Wg"],
                                         data["A"], data["Bt"], data["x0"], data["Z"], mode, T,
                                         seed, ws, want_intermediates=True)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    return {k: to_cpu(v) for k, v in res.items()}


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("mode", [binding.DFS_PATH_GREEDY, binding.DFS_PATH_VITERBI,
                                  binding.DFS_PATH_SAMPLE])
@pytest.mark.parametrize("T", [0.0, 0.8])
def test_fused_e4m3_small(lib, orc, spec, mode, T):
    data = wl.generate(spec, "cuda")
    npd = np_inputs(data)
    g = _run_e4m3(data, spec, mode, T, seed=spec.seed + 100)
    o = orc.select_verify(npd["h"], npd["W"], npd["Wg"], npd["A"], npd["Bt"], npd["x0"], npd["Z"],
                          path_mode=mode, temperature=T, seed=spec.seed + 100,
                          Wq=to_cpu(data["Wq"]), w_scale=to_cpu(data["w_scale"]))
    diverged = _compare(g, o, spec, list(range(spec.B)), T)
    assert diverged <= max(1, spec.B // 8)
    _invariants(g, spec, npd, T)


def test_fused_e4m3_full_size(lib, orc):
    """The E4M3 head at the throughput workload's full size, every request, greedy and the
    sampled traversal at T = 0.6."""
    spec = wl.THROUGHPUT.with_(lmhead="e4m3")
    data = wl.generate(spec, "cuda")
    npd = np_inputs(data)
    head = oracle_head(orc, npd, spec, Wq=to_cpu(data["Wq"]), w_scale=to_cpu(data["w_scale"]))
    for mode, T in ((binding.DFS_PATH_GREEDY, 0.0), (binding.DFS_PATH_SAMPLE, 0.6)):
        g = _run_e4m3(data, spec, mode, T, seed=spec.seed)
        _invariants(g, spec, npd, T)
        o = oracle_step(orc, npd, spec, head, mode, T, spec.seed)
        excluded = _compare(g, o, spec, range(spec.B), T,
                            name=f"{spec.name} e4m3 mode={mode} T={T}")
        assert excluded <= max(1, spec.B // 4)


@pytest.mark.parametrize("V,d", [(1000, 256), (4096, 128), (151936, 640)])
def test_pack_e4m3_head_layout(lib, V, d):
    """The packed head: tile (vb, kb) holds rows 128 vb .. 128 vb + 127 of Wq (zeros past V),
    bytes 128 kb .. 128 kb + 127 of each, as 16 KB contiguous; tiles by vb, then kb."""
    g = torch.Generator(device="cuda").manual_seed(V + d)
    Wq = torch.randint(0, 256, (V, d), generator=g, device="cuda", dtype=torch.uint8)
    got = binding.dfs_pack_e4m3_head(Wq)
    torch.cuda.synchronize()
    nvb, nkb = -(-V // 128), d // 128
    assert got.numel() == nvb * 128 * d
    pad = torch.zeros(nvb * 128, d, dtype=torch.uint8, device="cuda")
    pad[:V] = Wq
    want = pad.view(nvb, 128, nkb, 128).permute(0, 2, 1, 3).reshape(-1)
    assert torch.equal(got, want)
