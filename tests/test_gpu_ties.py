"""Exact logit ties planted in the LM head, inside the top-16 and exactly at its 16/17
boundary, on every LM-head kernel: the lower token id must win everywhere, both in the
order of the 16 candidates and in which of the tied tokens make the cut ("DFlash 2: Keep
Drafting Parallel", §"The right tokens are already there": the 16 best per position; the
tie rule is the library's, lower id first).

Construction (no near-tie rule applies: the tied logits are equal in fp32 and in fp64):
every hidden row has h[d-1] = 16; a base column w0 (bf16, w0[d-1] = 1) gives every row a
logit h . w0 near 16 (positive); 18 columns of W, spread over the vocabulary, are w0 scaled
by 2^e with e = 4, 4, 3, 3, 3, 2, 2, 1, 1, 1, 1, 0 x 7. A power-of-two scale is exact in
every product and partial sum, so columns with equal e have bit-identical logits on the
tensor cores and in the oracle, and even the smallest (e = 0) lies far above every other
logit of the row. The top-16 is then the 11 columns with e >= 1 and the 5 lowest ids of the
7 with e = 0."""
import math

import numpy as np
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl
from parity import close, to_cpu

pytestmark = pytest.mark.gpu

EXPONENTS = [4, 4, 3, 3, 3, 2, 2, 1, 1, 1, 1] + [0] * 7


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def _tie_inputs(B, L, V, d, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(B, L, d, generator=g)
    h[..., d - 1] = 16.0
    W = torch.randn(d, V, generator=g) / math.sqrt(d)
    w0 = (torch.randn(d, generator=g) / math.sqrt(d)).to(torch.bfloat16).float()
    w0[d - 1] = 1.0
    hot = torch.randperm(V, generator=g)[:len(EXPONENTS)]
    for e, v in zip(EXPONENTS, hot.tolist()):
        W[:, v] = w0 * 2.0 ** e  # exact in bf16
    return h.to(torch.bfloat16).contiguous(), W.to(torch.bfloat16).contiguous(), hot


def _expected_ids(hot):
    """The top-16 by (logit desc, id asc): groups by exponent, ids ascending in a group."""
    ids = []
    for e in (4, 3, 2, 1, 0):
        ids += sorted(int(v) for v, x in zip(hot.tolist(), EXPONENTS) if x == e)
    return ids[:16]


CASES = [  # (B, L, V, variant): <= 128 rows; CTA pairs, row-major and vocabulary-major
    (4, 8, 151936, "0"), (4, 8, 5000, "0"),
    (32, 8, 151936, "5"), (32, 8, 151936, "6"), (20, 9, 5000, "5"), (20, 9, 5000, "6"),
]


@pytest.mark.parametrize("B,L,V,variant", CASES)
def test_lmhead_ties_go_to_the_lower_id(lib, orc, B, L, V, variant, monkeypatch):
    monkeypatch.setenv("DFS_LMHEAD_VARIANT", variant)
    d = 256
    h, W, hot = _tie_inputs(B, L, V, d, seed=B * 1000 + V)
    want = _expected_ids(hot)
    # the oracle (fp64, exact ties) gives the same ids, in the same order, for every row
    rows = np.array([b * L + t for b in range(B) for t in range(1, L)])
    o_ids, o_U, _ = orc.topk(orc.logits(wl.to_numpy_bits(h), wl.to_numpy_bits(W), rows), 16)
    assert all(o_ids[i].tolist() == want for i in range(len(rows)))
    dims = binding.make_dims(B, L, V, d, 8, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    ids, U = binding.dfs_lmhead_topk(dims, h.cuda(), W.cuda(), ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    ids = to_cpu(ids).reshape(-1, 16)
    U = to_cpu(U).reshape(-1, 16)
    for i in range(len(rows)):
        assert ids[i].tolist() == want, f"row {i}: {ids[i].tolist()} != {want}"
        assert np.all(close(U[i], o_U[i]))
        # the tied logits are bit-identical on the GPU too
        for a, b in ((0, 1), (2, 3), (3, 4), (5, 6), (7, 8), (8, 9), (9, 10), (11, 15)):
            assert U[i, a] == U[i, b], f"row {i}: slots {a} and {b} not tied"


@pytest.mark.parametrize("B,L,V,variant", [(4, 8, 151936, "0"), (32, 8, 151936, "5"),
                                           (32, 8, 151936, "6")])
def test_fused_candidates_with_ties(lib, B, L, V, variant, monkeypatch):
    """The fused call's merge (inside the tail kernel) keeps the same tie order."""
    monkeypatch.setenv("DFS_LMHEAD_VARIANT", variant)
    d, r = 256, 16
    h, W, hot = _tie_inputs(B, L, V, d, seed=7 + B)
    want = _expected_ids(hot)
    g = torch.Generator().manual_seed(11)
    Wg = (torch.randn(r, d, generator=g) / math.sqrt(d)).to(torch.bfloat16).cuda()
    A = (torch.randn(V, r, generator=g) / math.sqrt(r)).to(torch.bfloat16).cuda()
    Bt = (torch.randn(V, r, generator=g) / math.sqrt(r)).to(torch.bfloat16).cuda()
    x0 = torch.randint(0, V, (B,), generator=g, dtype=torch.int32).cuda()
    Z = torch.randn(B, L, V, generator=g).to(torch.bfloat16).cuda()
    dims = binding.make_dims(B, L, V, d, r, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    res = binding.dfs_select_verify(dims, h.cuda(), W.cuda(), Wg, A, Bt, x0, Z,
                                    binding.DFS_PATH_GREEDY, 0.0, 1, ws, want_intermediates=True)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    ids = to_cpu(res["cand_ids"]).reshape(-1, 16)
    for i in range(ids.shape[0]):
        assert ids[i].tolist() == want, f"row {i}"


def _ramp_inputs(B, L, V, d):
    """Logits that grow with the token id, equal within each run of three consecutive ids."""
    g = torch.Generator().manual_seed(5)
    h = (torch.randn(B, L, d, generator=g) * 0.01).to(torch.bfloat16)
    h[..., d - 1] = 16.0
    h[..., d - 2] = 16.0
    ramp = torch.div(torch.arange(V), 3, rounding_mode="floor").double() * (12.0 / V)
    hi = ramp.to(torch.bfloat16)
    lo = (ramp - hi.double()).to(torch.bfloat16)
    W = torch.zeros(d, V, dtype=torch.bfloat16)
    W[d - 1] = hi
    W[d - 2] = lo
    return h, W


def _ramp_expected(V):
    """Five whole runs at the top and the lowest id of the sixth (lower id first in a run)."""
    top = V - 1 - (V - 1) % 3  # the first id of the highest run
    want = [top + k for k in range(V - top)]
    base = top
    while len(want) < 16:
        base -= 3
        want += [base + k for k in range(min(3, 16 - len(want)))]
    return want


@pytest.mark.parametrize("variant", ["5", "6"])
def test_lmhead_logits_increasing_with_id(lib, orc, variant, monkeypatch):
    """Logits that grow with the token id, equal within each run of three consecutive ids
    (every later tile beats every list, so every list is rebuilt on every tile). The top-16
    is five whole runs and the lowest id of the sixth: exact ties inside it and at its 16/17
    boundary, as the oracle gives them."""
    monkeypatch.setenv("DFS_LMHEAD_VARIANT", variant)
    B, L, V, d = 32, 8, 65528, 128
    h, W = _ramp_inputs(B, L, V, d)
    rows = np.array([b * L + t for b in range(B) for t in range(1, L)])
    o_ids, o_U, _ = orc.topk(orc.logits(wl.to_numpy_bits(h), wl.to_numpy_bits(W), rows), 16)
    dims = binding.make_dims(B, L, V, d, 8, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    ids, U = binding.dfs_lmhead_topk(dims, h.cuda(), W.cuda(), ws)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    ids = to_cpu(ids).reshape(-1, 16)
    U = to_cpu(U).reshape(-1, 16)
    want = _ramp_expected(V)
    assert all(o_ids[i].tolist() == want for i in range(len(rows)))
    for i in range(len(rows)):
        assert ids[i].tolist() == o_ids[i].tolist(), f"row {i}"
        assert np.all(close(U[i], o_U[i]))


@pytest.mark.parametrize("B,variant", [(4, "0"), (32, "5"), (32, "6")])
def test_fused_candidates_logits_increasing_with_id(lib, B, variant, monkeypatch):
    """The fused call's merge on the same ramp. The 16 lists with the best heads then hold
    far more entries above the 16th best head than its candidate buffer takes, so the merge
    takes its tree path; generic logits (the other tests) take the candidate ranks."""
    monkeypatch.setenv("DFS_LMHEAD_VARIANT", variant)
    L, V, d, r = 8, 65528, 128, 16
    h, W = _ramp_inputs(B, L, V, d)
    g = torch.Generator().manual_seed(13)
    Wg = (torch.randn(r, d, generator=g) / math.sqrt(d)).to(torch.bfloat16).cuda()
    A = (torch.randn(V, r, generator=g) / math.sqrt(r)).to(torch.bfloat16).cuda()
    Bt = (torch.randn(V, r, generator=g) / math.sqrt(r)).to(torch.bfloat16).cuda()
    x0 = torch.randint(0, V, (B,), generator=g, dtype=torch.int32).cuda()
    Z = torch.randn(B, L, V, generator=g).to(torch.bfloat16).cuda()
    dims = binding.make_dims(B, L, V, d, r, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    res = binding.dfs_select_verify(dims, h.cuda(), W.cuda(), Wg, A, Bt, x0, Z,
                                    binding.DFS_PATH_GREEDY, 0.0, 1, ws, want_intermediates=True)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    ids = to_cpu(res["cand_ids"]).reshape(-1, 16)
    want = _ramp_expected(V)
    for i in range(ids.shape[0]):
        assert ids[i].tolist() == want, f"row {i}"


@pytest.mark.parametrize("mode", [binding.DFS_PATH_GREEDY, binding.DFS_PATH_VITERBI])
@pytest.mark.parametrize("B,L,V,variant", [(4, 8, 5000, "0"), (32, 8, 151936, "5")])
def test_fused_path_ties_go_to_the_lower_id(lib, orc, B, L, V, variant, mode, monkeypatch):
    """Exact ties in the path choice of the fused call: with A = 0 every pair score is the
    successor's logit, S_t(a, c) = U_t(c) (exactly, on the GPU and in the oracle), and the
    planted logits tie the two best candidates of every position (e = 4). The greedy
    traversal's successor ties, and Viterbi's predecessor ties and final choice, must all go
    to the lower token id: the path is that token at every position. Compared with the
    oracle's path (its tie rule is pinned on the CPU) and its verification, request by
    request, with no near-tie exclusion."""
    monkeypatch.setenv("DFS_LMHEAD_VARIANT", variant)
    d, r = 256, 16
    h, W, hot = _tie_inputs(B, L, V, d, seed=23 + B)
    low4 = min(int(v) for v, e in zip(hot.tolist(), EXPONENTS) if e == 4)
    g = torch.Generator().manual_seed(19)
    Wg = (torch.randn(r, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    A = torch.zeros(V, r, dtype=torch.bfloat16)
    Bt = (torch.randn(V, r, generator=g) / math.sqrt(r)).to(torch.bfloat16)
    x0 = torch.randint(0, V, (B,), generator=g, dtype=torch.int32)
    Z = torch.randn(B, L, V, generator=g).to(torch.bfloat16)
    dims = binding.make_dims(B, L, V, d, r, binding.DFS_BF16, binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    res = binding.dfs_select_verify(dims, h.cuda(), W.cuda(), Wg.cuda(), A.cuda(), Bt.cuda(),
                                    x0.cuda(), Z.cuda(), mode, 0.0, 1, ws, want_intermediates=True)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    path, out, acc = to_cpu(res["path"]), to_cpu(res["out_tokens"]), to_cpu(res["accept_len"])
    cand_U = to_cpu(res["cand_U"]).reshape(B, L - 1, 16)
    assert np.all(cand_U[:, :, 0] == cand_U[:, :, 1])  # the planted tie reached the tail
    npd = {k: wl.to_numpy_bits(v) for k, v in (("h", h), ("W", W), ("Wg", Wg), ("A", A),
                                                 ("Bt", Bt), ("Z", Z))}
    rows = np.array([b * L + t for b in range(B) for t in range(1, L)])
    o_ids, o_U, _ = orc.topk(orc.logits(npd["h"], npd["W"], rows), 16)
    o_g = orc.gate(npd["h"], npd["Wg"], rows)
    fn = orc.path_viterbi if mode == binding.DFS_PATH_VITERBI else orc.path_greedy
    for b in range(B):
        sl = slice(b * (L - 1), (b + 1) * (L - 1))
        ids = o_ids[sl].reshape(L - 1, 16)
        S = orc.pair_scores(npd["A"], npd["Bt"], ids, o_U[sl].reshape(L - 1, 16),
                            o_g[sl].reshape(L - 1, -1), int(x0[b]))
        assert np.array_equal(S, np.broadcast_to(o_U[sl].reshape(L - 1, 1, 16), S.shape))
        o_path, _, o_score, _ = fn(S, ids)
        assert o_path.tolist() == [low4] * (L - 1), f"request {b}: oracle path"
        assert path[b].tolist() == [low4] * (L - 1), f"request {b}: path {path[b].tolist()}"
        o_out, o_acc = orc.verify_greedy(npd["Z"][b], o_path)
        assert acc[b] == o_acc and out[b].tolist() == o_out.tolist(), f"request {b}: verify"
