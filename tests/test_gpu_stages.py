"""GPU parity of each C-ABI stage against the fp64 oracle, stage-isolated: each GPU stage
is fed the oracle's upstream output so a failure points at one kernel.

Sizes span several vocabulary tiles with a ragged tail, one and two 128-row MMA tiles,
several 256-row groups, and the fp32 CUDA-core path."""
import numpy as np
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl
from parity import (ACC_MARGIN, GATE_ATOL, DRAW_MARGIN, PATH_MARGIN, close, compare_topk,
                    dims_for, np_inputs, to_cpu)

pytestmark = pytest.mark.gpu

SHAPES = [
    wl.TINY,  # fp32, CUDA-core path
    wl.TINY.with_(name="mt1_ragged", dtype="bf16", B=3, L=5, V=5000, d=512, r=64, seed=11),
    wl.TINY.with_(name="mt2_ragged", dtype="bf16", B=20, L=9, V=3000, d=256, r=32, seed=12),
    wl.TINY.with_(name="two_groups", dtype="bf16", B=40, L=8, V=2048, d=128, r=256, seed=13,
                  zipf=True),
    wl.TINY.with_(name="L2_minimal", dtype="bf16", B=2, L=2, V=1040, d=64, r=8, seed=14),
    wl.TINY.with_(name="L16_long", dtype="bf16", B=5, L=16, V=4096, d=192, r=128, seed=15),
]


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def _gen(spec):
    data = wl.generate(spec, "cuda")
    return data, np_inputs(data)


def _oracle_candidates(orc, npd, spec):
    B, L = spec.B, spec.L
    rows = np.array([b * L + t for b in range(B) for t in range(1, L)])
    u = orc.logits(npd["h"], npd["W"], rows)
    ids, U, gap = orc.topk(u, 16)
    P = L - 1
    return ids.reshape(B, P, 16), U.reshape(B, P, 16), gap.reshape(B, P), rows


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("variant", ["5", "6"])
def test_lmhead_topk(lib, orc, spec, variant, monkeypatch):
    monkeypatch.setenv("DFS_LMHEAD_VARIANT", variant)
    data, npd = _gen(spec)
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    ids, U = binding.dfs_lmhead_topk(dims, data["h"], data["W"], ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    o_ids, o_U, o_gap, _ = _oracle_candidates(orc, npd, spec)
    n, near, diverged = compare_topk(to_cpu(ids), to_cpu(U), o_ids, o_U, o_gap)
    assert diverged <= max(1, n // 50), f"{diverged}/{n} rows diverged on near-ties ({near} near)"


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
def test_pair_score_and_gate(lib, orc, spec):
    data, npd = _gen(spec)
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    o_ids, o_U, _, rows = _oracle_candidates(orc, npd, spec)
    U32 = o_U.astype(np.float32)
    ids_t = torch.from_numpy(o_ids.astype(np.int32)).cuda()
    U_t = torch.from_numpy(U32).cuda()
    S, gate = binding.dfs_pair_score(dims, data["h"], data["Wg"], data["A"], data["Bt"],
                                     data["x0"], ids_t, U_t, ws, want_gate=True)
    torch.cuda.synchronize()
    g_ref = orc.gate(npd["h"], npd["Wg"], rows).reshape(spec.B, spec.L - 1, spec.r)
    assert np.abs(to_cpu(gate) - g_ref).max() <= GATE_ATOL
    S_np = to_cpu(S)
    for b in range(spec.B):
        S_ref = orc.pair_scores(npd["A"], npd["Bt"], o_ids[b], U32[b].astype(np.float64), g_ref[b],
                                int(npd["x0"][b]))
        assert np.all(close(S_np[b], S_ref)), f"request {b}"


def _lattice(rng, B, P, mode):
    ids = np.stack([np.stack([rng.choice(50000, 16, replace=False) for _ in range(P)])
                    for _ in range(B)]).astype(np.int32)
    if mode == "ties":
        S = rng.integers(0, 3, (B, P, 16, 16)).astype(np.float32)  # exact in fp32: ties everywhere
    else:
        S = (rng.standard_normal((B, P, 16, 16)) * 3).astype(np.float32)
    S[:, 0, 1:, :] = S[:, 0, :1, :]
    return ids, S


@pytest.mark.parametrize("P", [1, 3, 7, 15])
@pytest.mark.parametrize("values", ["random", "ties"])
@pytest.mark.parametrize("mode", [binding.DFS_PATH_GREEDY, binding.DFS_PATH_VITERBI])
def test_path_select(lib, orc, P, values, mode):
    rng = np.random.default_rng(P * 10 + mode)
    B = 64
    ids, S = _lattice(rng, B, P, values)
    dims = binding.make_dims(B, P + 1, 50000, 64, 8, 0, 0)
    path, score = binding.dfs_path_select(dims, torch.from_numpy(S).cuda(),
                                          torch.from_numpy(ids).cuda(), mode)
    torch.cuda.synchronize()
    path, score = to_cpu(path), to_cpu(score)
    fn = orc.path_viterbi if mode == binding.DFS_PATH_VITERBI else orc.path_greedy
    diverged = 0
    for b in range(B):
        o_path, _, o_score, margin = fn(S[b].astype(np.float64), ids[b])
        if path[b].tolist() != o_path.tolist():
            # integer lattices are exact in fp32, so ties must be broken identically there
            assert values == "random" and margin < PATH_MARGIN, f"request {b}: path differs"
            diverged += 1
            continue
        assert close(score[b], o_score)
    assert diverged <= B // 16


def _planted_path(rng, Z, L, agree):
    y = np.argmax(Z.astype(np.float64), axis=-1)
    path = y[:, :L - 1].copy()
    flip = rng.random(path.shape) > agree
    path[flip] = (path[flip] + 1 + rng.integers(0, 100, flip.sum())) % Z.shape[-1]
    return path.astype(np.int32)


@pytest.mark.parametrize("zdtype", ["bf16", "fp32"])
@pytest.mark.parametrize("L,V", [(8, 5000), (2, 1024), (16, 20000)])
def test_verify_greedy(lib, orc, zdtype, L, V):
    rng = np.random.default_rng(L + V)
    B = 24
    Zf = np.round(rng.standard_normal((B, L, V)) * 4) / 4  # coarse values: exact ties at the max
    Zt = torch.from_numpy(Zf.astype(np.float32)).cuda()
    if zdtype == "bf16":
        Zt = Zt.to(torch.bfloat16)
    Znp = wl.to_numpy_bits(Zt)
    Zref = Zt.float().cpu().numpy()
    path = _planted_path(rng, Zref, L, 0.8)
    code = binding.DFS_BF16 if zdtype == "bf16" else binding.DFS_FP32
    dims = binding.make_dims(B, L, V, 64, 8, code, code)
    ws = binding.alloc_workspace(dims)
    out, acc = binding.dfs_verify(dims, torch.from_numpy(path).cuda(), Zt, 0.0, 0, ws)
    torch.cuda.synchronize()
    out, acc = to_cpu(out), to_cpu(acc)
    for b in range(B):
        o_out, o_acc = orc.verify_greedy(Znp[b], path[b])
        assert acc[b] == o_acc and out[b].tolist() == o_out.tolist(), f"request {b}"


@pytest.mark.parametrize("T", [0.6, 1.0, 2.5])
@pytest.mark.parametrize("L,V", [(8, 9000), (4, 1024), (16, 30000)])
def test_verify_sampling(lib, orc, T, L, V):
    rng = np.random.default_rng(int(T * 10) + L + V)
    B = 48
    Zt = (torch.from_numpy(rng.standard_normal((B, L, V)).astype(np.float32)) * 3).cuda()
    Zt = Zt.to(torch.bfloat16)
    Znp = wl.to_numpy_bits(Zt)
    path = _planted_path(rng, Zt.float().cpu().numpy(), L, 0.9)
    dims = binding.make_dims(B, L, V, 64, 8, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    seed = 1234 + L
    out, acc = binding.dfs_verify(dims, torch.from_numpy(path).cuda(), Zt, T, seed, ws)
    torch.cuda.synchronize()
    out, acc = to_cpu(out), to_cpu(acc)
    diverged = 0
    for b in range(B):
        o_out, o_acc, am, gm = orc.verify_sampling(Znp[b], path[b], T, seed, b=b)
        if acc[b] != o_acc or out[b].tolist() != o_out.tolist():
            assert am < ACC_MARGIN or gm < DRAW_MARGIN, f"request {b}: differs without a near-tie"
            diverged += 1
    assert diverged <= B // 16


def test_verify_greedy_more_rows_than_one_grid_dimension(lib):
    """More target rows than the 65535 blocks of a grid's second dimension (4375 requests of
    16 positions = 70000 rows over a 4096-token vocabulary): the row statistics still cover
    every row. Every request is checked against target-argmax decoding of its rows, which
    greedy verification must reproduce token for token."""
    rng = np.random.default_rng(70000)
    B, L, V = 4375, 16, 4096
    Zt = (torch.randn(B, L, V, device="cuda", generator=torch.Generator("cuda").manual_seed(3))
          * 3).to(torch.bfloat16)
    y = Zt.float().argmax(-1)  # lower id on ties, as the library's rule
    path = y[:, :L - 1].clone()
    flip = torch.from_numpy(rng.random((B, L - 1)) > 0.9).cuda()
    path[flip] = (path[flip] + 1) % V
    path = path.to(torch.int32).contiguous()
    dims = binding.make_dims(B, L, V, 64, 8, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    out, acc = binding.dfs_verify(dims, path, Zt, 0.0, 0, ws)
    torch.cuda.synchronize()
    y, path, out, acc = to_cpu(y), to_cpu(path), to_cpu(out), to_cpu(acc)
    agree = path == y[:, :L - 1]
    n = np.where(agree.all(1), L - 1, np.argmin(agree, axis=1))  # leading agreements
    assert np.array_equal(acc, n + 1)
    for b in range(B):
        assert out[b, :n[b]].tolist() == path[b, :n[b]].tolist()
        assert out[b, n[b]] == y[b, n[b]] and np.all(out[b, n[b] + 1:] == -1)
