"""Pins for the sampled-traversal proposal and its speculative-sampling verification
(oracle.cpp: orc_path_sample, orc_verify_proposal), checked against what the method and the
mathematics fix rather than against the oracle itself:

  * the sampled path's distribution is the product of the per-step softmaxes of the scores
    ("sampling draws from the same scores", [Blog] "A lightweight path selector");
  * each emitted token is distributed as the target's softmax given the tokens before it
    (rejection sampling recovers the exact target distribution, [Blog] ibid.; Leviathan
    et al. 2023), for a proposal deliberately unlike the target;
  * the probability of accepting the first draft is sum_v min(p(v), q(v));
  * a proposal with all its mass on one token reproduces the deterministic-proposal
    verification token for token; T -> 0 reduces to the greedy traversal and verification.
"""
import numpy as np
import pytest
from scipy import stats

import oracle as orc_mod

T = 0.8


def _softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def _chisq_p(counts, expected):
    """Chi-square p-value after merging the cells with expected count < 5 into one."""
    counts = np.asarray(counts, np.float64)
    expected = np.asarray(expected, np.float64)
    small = expected < 5
    if small.any():
        counts = np.append(counts[~small], counts[small].sum())
        expected = np.append(expected[~small], expected[small].sum())
    return stats.chisquare(counts, expected * counts.sum() / expected.sum()).pvalue


def _lattice(rng, P, K, V, scale=1.5):
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(P)]).astype(np.int32)
    S = rng.standard_normal((P, K, K)) * scale
    S[0, 1:, :] = S[0, :1, :]  # position 1's predecessor is the last verified token
    return S, ids


def test_sampled_path_distribution(orc):
    rng = np.random.default_rng(7)
    P, K, V = 2, 16, 200
    S, ids = _lattice(rng, P, K, V)
    Z = rng.standard_normal((P + 1, V)).astype(np.float32)
    n = 200_000
    paths, _, _ = orc.sample_verify_many(Z, S, ids, T, 1000, n)
    pos = {int(t): i for i, t in enumerate(ids[0])}, {int(t): i for i, t in enumerate(ids[1])}
    a = np.array([pos[0][int(x)] for x in paths[:, 0]])
    c = np.array([pos[1][int(x)] for x in paths[:, 1]])
    counts = np.bincount(a * K + c, minlength=K * K)
    q1 = _softmax(S[0, 0] / T)
    expected = np.concatenate([q1[i] * _softmax(S[1, i] / T) for i in range(K)]) * n
    assert _chisq_p(counts, expected) > 0.01


def _proposal_case(seed, L, V=64, K=16):
    rng = np.random.default_rng(seed)
    S, ids = _lattice(rng, L - 1, K, V, scale=2.0)
    Z = (rng.standard_normal((L, V)) * 1.5).astype(np.float32)
    return S, ids, Z


def test_first_token_is_target_distributed(orc):
    S, ids, Z = _proposal_case(11, L=2)
    n = 400_000
    _, out, acc = orc.sample_verify_many(Z, S, ids, T, 5_000, n)
    p0 = _softmax(Z[0].astype(np.float64) / T)
    q = np.zeros_like(p0)
    q[ids[0]] = _softmax(S[0, 0] / T)
    assert np.abs(p0 - q).sum() > 0.5  # the proposal really differs from the target
    counts = np.bincount(out[:, 0], minlength=Z.shape[1])
    assert _chisq_p(counts, p0 * n) > 0.01


def test_second_token_is_target_distributed(orc):
    S, ids, Z = _proposal_case(12, L=3)
    n = 400_000
    _, out, acc = orc.sample_verify_many(Z, S, ids, T, 9_000, n)
    emitted = acc >= 2
    p1 = _softmax(Z[1].astype(np.float64) / T)
    counts = np.bincount(out[emitted, 1], minlength=Z.shape[1])
    assert emitted.sum() > 1000
    assert _chisq_p(counts, p1 * emitted.sum()) > 0.01


def test_first_acceptance_rate_closed_form(orc):
    S, ids, Z = _proposal_case(13, L=2)
    n = 200_000
    _, _, acc = orc.sample_verify_many(Z, S, ids, T, 77, n)
    p0 = _softmax(Z[0].astype(np.float64) / T)
    q1 = _softmax(S[0, 0] / T)
    rate = np.minimum(p0[ids[0]], q1).sum()
    got = (acc == 2).mean()
    assert abs(got - rate) < 4 * np.sqrt(rate * (1 - rate) / n)


def test_point_mass_proposal_is_the_deterministic_verification(orc):
    rng = np.random.default_rng(21)
    L, V, K = 5, 300, 16
    S, ids = _lattice(rng, L - 1, K, V)
    S[:, :, 3] += 5000.0  # q puts all its mass (exactly 1 in fp64) on candidate 3
    Z = rng.standard_normal((L, V)).astype(np.float32)
    for seed in range(200):
        path, pidx, q, _, _ = orc.path_sample(S, ids, T, seed)
        assert np.all(pidx == 3) and np.all(q[:, 3] == 1.0)
        a = orc.verify_proposal(Z, path, ids, q, pidx, T, seed)
        b = orc.verify_sampling(Z, path, T, seed)
        if min(a[3], b[3]) < 1e-9:  # the redraws' weights differ by a constant factor: near-ties
            continue
        assert a[0].tolist() == b[0].tolist() and a[1] == b[1]


def test_zero_temperature_is_greedy(orc):
    from draft_speculative_decoding_gb300 import workloads as wl
    spec = wl.TINY.with_(name="t0", B=2, L=4, V=512, d=64, r=16, seed=3)
    data = wl.generate(spec, "cpu")
    npd = {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}
    args = [npd[k] for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")]
    g = orc.select_verify(*args, path_mode=0, temperature=0.0, seed=5)
    s = orc.select_verify(*args, path_mode=2, temperature=0.0, seed=5)
    for k in ("path", "out_tokens", "accept_len"):
        assert np.array_equal(g[k], s[k]), k


def test_whole_step_composes_the_stages(orc):
    from draft_speculative_decoding_gb300 import workloads as wl
    spec = wl.TINY.with_(name="comp", B=3, L=5, V=700, d=64, r=16, seed=4)
    data = wl.generate(spec, "cpu")
    npd = {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}
    res = orc.select_verify(*[npd[k] for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")],
                            path_mode=2, temperature=T, seed=9)
    Z = npd["Z"].reshape(spec.B, spec.L, spec.V)
    for b in range(spec.B):
        path, pidx, q, score, _ = orc.path_sample(res["S"][b], res["cand_ids"][b], T, 9, b)
        assert path.tolist() == res["path"][b].tolist()
        assert score == pytest.approx(res["path_score"][b])
        out, acc, _, _ = orc.verify_proposal(Z[b], path, res["cand_ids"][b], q, pidx, T, 9, b)
        assert out.tolist() == res["out_tokens"][b].tolist() and acc == res["accept_len"][b]
