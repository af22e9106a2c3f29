"""Pins for the joint path draw (oracle.cpp: orc_path_sample_joint): a draw of the whole path
from the distribution the pair scores define over the lattice, P(x_1..x_P) proportional to
exp(sum_t S_t(x_{t-1}, x_t) / T) ("DFlash 2: Keep Drafting Parallel", §"A lightweight path
selector": sampling draws from the same scores; rejection sampling recovers the target).
Checked against brute force over every path of small lattices, not against the oracle:

  * each conditional the draw reports is the exact conditional of the joint distribution
    given the drawn prefix, so their product along the path is the path's probability;
  * the frequencies of drawn paths follow the joint distribution (chi-square);
  * T -> 0 gives the max-sum (Viterbi) path;
  * verified against its own conditionals, every emitted token is target-distributed.
"""
import itertools

import numpy as np
import pytest
from scipy import stats

from test_oracle_proposal import _chisq_p, _lattice, _softmax


def _brute_force(S, T):
    """Every path as candidate indices, and its exact probability under the joint."""
    P, K, _ = S.shape
    paths = np.array(list(itertools.product(range(K), repeat=P)))
    score = S[0, 0, paths[:, 0]].copy()
    for p in range(1, P):
        score += S[p, paths[:, p - 1], paths[:, p]]
    return paths, _softmax(score / T), score


@pytest.mark.parametrize("T", [0.7, 1.5])
def test_conditionals_are_exact_and_multiply_to_the_path_probability(orc, T):
    rng = np.random.default_rng(int(T * 10))
    P, K, V = 3, 16, 500
    S, ids = _lattice(rng, P, K, V)
    paths, prob, _ = _brute_force(S, T)
    for seed in range(40):
        path, pidx, q, score, _ = orc.path_sample_joint(S, ids, T, seed, b=3)
        assert path.tolist() == [int(ids[p, pidx[p]]) for p in range(P)]
        for p in range(P):  # the conditional given the drawn prefix, by brute force
            prefix = np.all(paths[:, :p] == pidx[:p], axis=1)
            cond = np.array([prob[prefix & (paths[:, p] == c)].sum() for c in range(K)])
            np.testing.assert_allclose(q[p], cond / cond.sum(), rtol=1e-10, atol=1e-15)
        row = np.all(paths == pidx, axis=1)
        np.testing.assert_allclose(np.prod(q[np.arange(P), pidx]), prob[row][0], rtol=1e-10)
        assert score == pytest.approx(S[0, 0, pidx[0]] + sum(S[p, pidx[p - 1], pidx[p]]
                                                              for p in range(1, P)))


def test_drawn_path_frequencies_follow_the_joint(orc):
    rng = np.random.default_rng(3)
    P, K, V, T = 2, 16, 200, 0.9
    S, ids = _lattice(rng, P, K, V)
    Z = rng.standard_normal((P + 1, V)).astype(np.float32)
    n = 200_000
    drawn, _, _ = orc.sample_verify_many(Z, S, ids, T, 2000, n, joint=True)
    col = [{int(t): i for i, t in enumerate(ids[p])} for p in range(P)]
    idx = np.array([[col[p][int(x)] for p, x in enumerate(row)] for row in drawn])
    counts = np.bincount(idx[:, 0] * K + idx[:, 1], minlength=K * K)
    paths, prob, _ = _brute_force(S, T)
    assert _chisq_p(counts, prob[np.argsort(paths[:, 0] * K + paths[:, 1])] * n) > 0.01
    # it is not the left-to-right traversal's distribution (which ignores the later scores)
    q1 = _softmax(S[0, 0] / T)
    trav = np.concatenate([q1[i] * _softmax(S[1, i] / T) for i in range(K)])
    assert np.abs(trav - prob[np.argsort(paths[:, 0] * K + paths[:, 1])]).sum() > 0.05


def test_low_temperature_is_the_viterbi_path(orc):
    rng = np.random.default_rng(8)
    for _ in range(20):
        P, K = 5, 16
        S, ids = _lattice(rng, P, K, 1000, scale=3.0)
        v_path, _, _, _ = orc.path_viterbi(S, ids)
        j_path, _, _, _, _ = orc.path_sample_joint(S, ids, 1e-4, int(rng.integers(1 << 30)))
        assert j_path.tolist() == v_path.tolist()


@pytest.mark.parametrize("pos", [0, 1])
def test_emitted_tokens_are_target_distributed(orc, pos):
    rng = np.random.default_rng(21 + pos)
    L, V, K, T = 3, 64, 16, 0.8
    S, ids = _lattice(rng, L - 1, K, V, scale=2.0)
    Z = (rng.standard_normal((L, V)) * 1.5).astype(np.float32)
    n = 400_000
    _, out, acc = orc.sample_verify_many(Z, S, ids, T, 70_000, n, joint=True)
    emitted = acc >= pos + 1
    p = _softmax(Z[pos].astype(np.float64) / T)
    counts = np.bincount(out[emitted, pos], minlength=V)
    assert emitted.sum() > 1000
    assert _chisq_p(counts, p * emitted.sum()) > 0.01
