"""The oracle's whole-step function against its own stages and brute force, on the
tiny workload (fp32, B=1, L=4, V=1024, d=256, r=32) and a ragged bf16 case."""
import numpy as np
import pytest

from draft_speculative_decoding_gb300 import workloads as wl
from test_oracle_pair_path import _brute_force


def _np(data):
    return {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}


@pytest.mark.parametrize("spec", [
    wl.TINY,
    wl.TINY.with_(name="ragged_bf16", dtype="bf16", B=3, L=5, V=2056, d=128, r=48, seed=21,
                  zipf=True),
])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T", [0.0, 0.7])
def test_select_verify_composes_stages(orc, spec, mode, T):
    data = _np(wl.generate(spec))
    res = orc.select_verify(data["h"], data["W"], data["Wg"], data["A"], data["Bt"], data["x0"],
                            data["Z"], path_mode=mode, temperature=T, seed=spec.seed)
    B, L = spec.B, spec.L
    for q in range(B):
        rows = q * L + np.arange(1, L)
        u = orc.logits(data["h"], data["W"], rows)
        ids, U, gap = orc.topk(u, 16)
        np.testing.assert_array_equal(res["cand_ids"][q], ids)
        np.testing.assert_array_equal(res["cand_U"][q], U)
        g = orc.gate(data["h"], data["Wg"], rows)
        np.testing.assert_array_equal(res["gate"][q], g)
        S = orc.pair_scores(data["A"], data["Bt"], ids, U, g, int(data["x0"][q]))
        np.testing.assert_array_equal(res["S"][q], S)
        fn = orc.path_viterbi if mode == 1 else orc.path_greedy
        path, _, score, _ = fn(S, ids)
        assert res["path"][q].tolist() == path.tolist() and res["path_score"][q] == score
        if mode == 1 and L - 1 <= 3:
            assert _brute_force(S, ids)[0] == path.tolist()
        if T > 0:
            out, acc, _, _ = orc.verify_sampling(data["Z"][q], path, T, spec.seed, b=q)
        else:
            out, acc = orc.verify_greedy(data["Z"][q], path)
        assert res["out_tokens"][q].tolist() == out.tolist() and res["accept_len"][q] == acc


def test_select_verify_request_subset(orc):
    spec = wl.TINY.with_(name="subset", dtype="bf16", B=4, L=3, V=512, d=64, r=16, seed=5)
    data = _np(wl.generate(spec))
    full = orc.select_verify(*(data[k] for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")),
                             path_mode=1, temperature=1.0, seed=3)
    sub = orc.select_verify(*(data[k] for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")),
                            path_mode=1, temperature=1.0, seed=3, reqs=[2, 0])
    for key in ("cand_ids", "path", "out_tokens", "accept_len"):
        np.testing.assert_array_equal(sub[key], full[key][[2, 0]])


@pytest.mark.parametrize("mode,T", [(0, 0.0), (1, 0.0), (0, 0.7), (1, 1.3), (2, 0.7), (3, 0.7),
                                    (3, 0.0)])
def test_stagewise_oracle_step_equals_select_verify(orc, mode, T):
    """The GPU tests compose the oracle's step from its stages on a head computed once per
    workload (tests/parity.py: oracle_head, oracle_step); that composition must equal the
    oracle's own whole step."""
    from parity import oracle_head, oracle_step
    spec = wl.TINY.with_(name="stagewise", dtype="bf16", B=5, L=6, V=900, d=128, r=16, seed=8)
    data = wl.generate(spec, "cpu")
    npd = {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}
    ref = orc.select_verify(*[npd[k] for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")],
                            path_mode=mode, temperature=T, seed=21)
    got = oracle_step(orc, npd, spec, oracle_head(orc, npd, spec), mode, T, 21)
    for k in ("cand_ids", "cand_U", "topk_gap", "S", "path", "path_score", "path_margin",
              "out_tokens", "accept_len", "acc_margin", "draw_margin"):
        assert np.array_equal(np.asarray(got[k]), np.asarray(ref[k])), k
