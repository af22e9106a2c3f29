"""Pins for the oracle's pair scores and path selection.

Pair scores: a hand-derived lattice (tests/golden/pair_path_example.json),
one-hot closed forms, linearity, and the A = 0 reduction to unigram scores.
Viterbi: brute force over every path. Greedy: the hand-derived lattice where
greedy and Viterbi part ways, and the A = 0 reduction to top-1 per position."""
import itertools
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "pair_path_example.json")) as f:
        return json.load(f)


def test_pair_scores_hand_worked_example(orc):
    gd = _golden()
    A = np.array(gd["A"], np.float32)
    Bt = np.array(gd["B"], np.float32)
    S = orc.pair_scores(A, Bt, np.array(gd["ids"]), np.array(gd["U"]), np.array(gd["gate"]),
                        gd["x0"])
    np.testing.assert_array_equal(S, np.array(gd["S"]))


def test_paths_hand_worked_example(orc):
    gd = _golden()
    S = np.array(gd["S"], np.float64)
    ids = np.array(gd["ids"], np.int32)
    gp, _, gs, _ = orc.path_greedy(S, ids)
    vp, _, vs, _ = orc.path_viterbi(S, ids)
    assert gp.tolist() == gd["greedy_path"] and gs == gd["greedy_score"]
    assert vp.tolist() == gd["viterbi_path"] and vs == gd["viterbi_score"]


def test_pair_scores_one_hot_closed_form(orc):
    # A(a) = e_{i(a)}, B(b) = e_{j(b)}, gate = c_j: S(a,b) = U(b) + c_{i(a)} [i(a) == j(b)]
    V, r, K, P = 40, 8, 4, 3
    rng = np.random.default_rng(11)
    ia = rng.integers(0, r, V)
    jb = rng.integers(0, r, V)
    A = np.zeros((V, r), np.float32)
    Bt = np.zeros((V, r), np.float32)
    A[np.arange(V), ia] = 1
    Bt[np.arange(V), jb] = 1
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(P)]).astype(np.int32)
    U = rng.standard_normal((P, K))
    g = rng.uniform(0.1, 0.9, (P, r))
    x0 = 17
    S = orc.pair_scores(A, Bt, ids, U, g, x0)
    for p in range(P):
        for a in range(K):
            ta = x0 if p == 0 else ids[p - 1, a]
            for b in range(K):
                tb = ids[p, b]
                bonus = g[p, ia[ta]] if ia[ta] == jb[tb] else 0.0
                assert S[p, a, b] == U[p, b] + bonus


def test_pair_scores_linear_in_tables_and_gate(orc):
    V, r, K, P = 30, 16, 16, 2
    rng = np.random.default_rng(5)
    # multiples of 1/16 keep A1 + A2 exact in fp32
    A1, A2, Bt = (np.round(rng.standard_normal((V, r)) * 16).astype(np.float32) / 16
                  for _ in range(3))
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(P)]).astype(np.int32)
    U = rng.standard_normal((P, K))
    g = rng.uniform(0, 1, (P, r))
    S1 = orc.pair_scores(A1, Bt, ids, U, g, 3)
    S2 = orc.pair_scores(A2, Bt, ids, U, g, 3)
    S12 = orc.pair_scores(A1 + A2, Bt, ids, U, g, 3)
    np.testing.assert_allclose(S12 - U[:, None, :], (S1 - U[:, None, :]) + (S2 - U[:, None, :]),
                               rtol=1e-12, atol=1e-12)
    Sg = orc.pair_scores(A1, Bt, ids, U, 2 * g, 3)
    np.testing.assert_allclose(Sg - U[:, None, :], 2 * (S1 - U[:, None, :]), rtol=1e-12, atol=1e-12)
    # position 1 reads the last verified token: all of its a-rows coincide
    assert np.all(S1[0] == S1[0, :1])


def test_zero_tables_reduce_to_top1(orc):
    V, r, K, P = 50, 4, 16, 5
    rng = np.random.default_rng(2)
    A = np.zeros((V, r), np.float32)
    Bt = rng.standard_normal((V, r)).astype(np.float32)
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(P)]).astype(np.int32)
    U = -np.sort(-rng.standard_normal((P, K)), axis=1)  # candidate lists ordered by U desc
    S = orc.pair_scores(A, Bt, ids, U, rng.uniform(0, 1, (P, r)), 9)
    assert np.all(S == U[:, None, :])
    for fn in (orc.path_greedy, orc.path_viterbi):
        path, pidx, _, _ = fn(S, ids)
        assert pidx.tolist() == [0] * P
        assert path.tolist() == ids[:, 0].tolist()


def _brute_force(S, ids):
    """Every path scored left to right; best value, ties -> smallest reversed token tuple."""
    P, K, _ = S.shape
    best = None
    for combo in itertools.product(range(K), repeat=P):
        tot = S[0, 0, combo[0]]
        for p in range(1, P):
            tot = tot + S[p, combo[p - 1], combo[p]]
        toks = tuple(int(ids[p, combo[p]]) for p in range(P))
        key = (-tot, toks[::-1])
        if best is None or key < best[0]:
            best = (key, toks, tot)
    return list(best[1]), best[2]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("P,K", [(3, 16), (4, 6), (2, 16)])
def test_viterbi_equals_brute_force(orc, seed, P, K):
    rng = np.random.default_rng(100 * seed + P)
    ids = np.stack([rng.choice(1000, K, replace=False) for _ in range(P)]).astype(np.int32)
    S = np.round(rng.standard_normal((P, K, K)), 1 if seed % 2 else 6)  # coarse rounding plants ties
    S[0, 1:] = S[0, :1]
    path, _, score, _ = orc.path_viterbi(S, ids)
    ref_path, ref_score = _brute_force(S, ids)
    assert path.tolist() == ref_path
    assert score == ref_score


def test_greedy_is_stepwise_best_successor(orc):
    # on a lattice built so each step's best successor is unique, greedy follows it
    rng = np.random.default_rng(4)
    P, K = 6, 16
    ids = np.stack([rng.choice(500, K, replace=False) for _ in range(P)]).astype(np.int32)
    S = rng.standard_normal((P, K, K))
    S[0, 1:] = S[0, :1]
    path, pidx, score, _ = orc.path_greedy(S, ids)
    a, tot = 0, 0.0
    for p in range(P):
        b = int(np.argmax(S[p, a]))
        assert pidx[p] == b
        tot += S[p, a, b]
        a = b
    assert score == tot
    # ties at a step: the lower token id wins
    S2 = np.zeros((1, K, K))
    ids2 = np.array([[9, 4, 7] + list(range(100, 100 + K - 3))], np.int32)
    p2, _, _, margin = orc.path_greedy(S2, ids2)
    assert p2.tolist() == [4] and margin == 0.0


def test_paths_shift_invariant(orc):
    rng = np.random.default_rng(8)
    P, K = 5, 16
    ids = np.stack([rng.choice(900, K, replace=False) for _ in range(P)]).astype(np.int32)
    S = rng.standard_normal((P, K, K))
    S[0, 1:] = S[0, :1]
    shift = np.array([0.5, -2.0, 8.0, 0.25, -1.0])[:, None, None]  # per-position constants (exact)
    for fn in (orc.path_greedy, orc.path_viterbi):
        assert fn(S, ids)[0].tolist() == fn(S + shift, ids)[0].tolist()


@pytest.mark.parametrize("seed", range(8))
def test_viterbi_equals_brute_force_on_tie_heavy_lattices(orc, seed):
    # integer scores in {0, 1, 2}: equal path totals and equal predecessor values everywhere
    rng = np.random.default_rng(500 + seed)
    P, K = 3, 8
    ids = np.stack([rng.choice(60, K, replace=False) for _ in range(P)]).astype(np.int32)
    S = rng.integers(0, 3, (P, K, K)).astype(np.float64)
    S[0, 1:] = S[0, :1]
    assert orc.path_viterbi(S, ids)[0].tolist() == _brute_force(S, ids)[0]


def test_viterbi_predecessor_tie_goes_to_lower_token_id(orc):
    # delta_1 = (1, 1, 0) over tokens (50, 10, 30); S_2 = 0: every final state is reached
    # equally well from token 50 (index 0) and token 10 (index 1); token 10 must win.
    ids = np.array([[50, 10, 30], [7, 3, 5]], np.int32)
    S = np.zeros((2, 3, 3))
    S[0, :, :] = [1.0, 1.0, 0.0]
    path, pidx, score, margin = orc.path_viterbi(S, ids)
    assert path.tolist() == [10, 3] and pidx.tolist() == [1, 1] and score == 1.0 and margin == 0.0
