"""Pins for the oracle's verification and random numbers.

Greedy verification is pinned to target-argmax (autoregressive) decoding via
numpy argmax. Sampling verification is pinned by chi-square tests of the
emitted-token distributions against the target softmax (the pages' claim that
rejection sampling keeps the target distribution) and by limiting cases.
Philox4x64-10 is pinned to numpy.random.Philox. The accept-length definition is
pinned to the verify lengths printed in the blog's Table 1."""
import itertools
import json
import os

import numpy as np
import pytest
from scipy import stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- Philox4x64-10
@pytest.mark.parametrize("ctr,key", [
    ([1, 0, 0, 0], [1, 2]),
    ([0x0123456789ABCDEF, 7, 2**63 + 5, 99], [2**64 - 1, 12345]),
    ([5, 3, 31, 1], [20260818, 0]),
])
def test_philox_matches_numpy(orc, ctr, key):
    # numpy's Philox advances its counter before producing a block, so a numpy
    # generator whose counter is (ctr - 1) emits the block for ctr first.
    c = int(ctr[0]) | (int(ctr[1]) << 64) | (int(ctr[2]) << 128) | (int(ctr[3]) << 192)
    c -= 1
    words = [(c >> (64 * i)) & (2**64 - 1) for i in range(4)]
    g = np.random.Philox(key=np.array(key, np.uint64), counter=np.array(words, np.uint64))
    expect = g.random_raw(4).astype(np.uint64)
    np.testing.assert_array_equal(orc.philox4x64(ctr, key), expect)


# ---------------------------------------------------------------- greedy verify
def _ar_decode(Z, path):
    """Target-argmax decoding: keep drafting tokens while they equal the target's argmax."""
    L = Z.shape[0]
    out = []
    for i in range(L):
        y = int(np.argmax(Z[i]))  # first maximum = lower id
        out.append(y)
        if i == L - 1 or path[i] != y:
            break
    return out


@pytest.mark.parametrize("seed", range(40))
def test_greedy_verify_equals_target_argmax_decoding(orc, seed):
    rng = np.random.default_rng(seed)
    L, V = int(rng.integers(2, 17)), int(rng.integers(16, 300))
    Z = np.round(rng.standard_normal((L, V)), 1).astype(np.float32)  # coarse: ties happen
    y = np.argmax(Z, axis=1)
    path = y[:L - 1].copy()
    cut = int(rng.integers(0, L))  # plant the first mismatch at position cut+1 (none if cut == L-1)
    if cut < L - 1:
        path[cut] = (path[cut] + 1 + int(rng.integers(0, V - 1))) % V
    out, acc = orc.verify_greedy(Z, path)
    ref = _ar_decode(Z, path)
    assert acc == len(ref) == min(cut, L - 1) + 1
    assert out[:acc].tolist() == ref
    assert np.all(out[acc:] == -1)


def test_greedy_verify_full_and_zero_acceptance(orc):
    rng = np.random.default_rng(1)
    Z = rng.standard_normal((8, 64)).astype(np.float32)
    y = np.argmax(Z, 1)
    out, acc = orc.verify_greedy(Z, y[:7])
    assert acc == 8 and out.tolist() == y.tolist()
    bad = y[:7].copy()
    bad[0] = (bad[0] + 1) % 64
    out, acc = orc.verify_greedy(Z, bad)
    assert acc == 1 and out[0] == y[0]


# ---------------------------------------------- accept length vs the blog's Table 1
def test_accept_length_reproduces_blog_table1(orc):
    """Verify length = 1 + sum_k prod_{j<=k} r_j, with r_j the per-position recall
    conditioned on earlier positions being correct. Enumerate all 2^7 agreement patterns
    through the oracle's greedy verification; the exact expectation must equal the
    verify lengths printed beside the recall rows (to the printed precision)."""
    with open(os.path.join(GOLDEN, "blog_table1_recall.json")) as f:
        gd = json.load(f)
    P, V = gd["positions"], 32
    L = P + 1
    Z = np.zeros((L, V), np.float32)
    for i in range(L):
        Z[i, i] = 1.0  # target argmax of row i is token i
    for key, printed in (("recall_at_1", gd["verify_length_recall_at_1"]),
                         ("recall_at_16", gd["verify_length_recall_at_16"])):
        r = np.array(gd[key])
        expect = 0.0
        for pattern in itertools.product([0, 1], repeat=P):
            prob = np.prod([r[j] if pattern[j] else 1 - r[j] for j in range(P)])
            path = np.array([j if pattern[j] else V - 1 - j for j in range(P)], np.int32)
            _, acc = orc.verify_greedy(Z, path)
            expect += prob * acc
        closed = 1 + sum(np.prod(r[:k + 1]) for k in range(P))
        assert abs(expect - closed) < 1e-12
        assert abs(expect - printed) <= gd["printed_precision"] + 1e-9


# ---------------------------------------------------------------- sampling verify
def _softmax(z, T):
    x = z.astype(np.float64) / T
    x -= x.max()
    e = np.exp(x)
    return e / e.sum()


def _chi2_pvalue(counts, probs):
    n = counts.sum()
    exp = probs * n
    order = np.argsort(exp)
    # merge the smallest-expectation bins until each merged bin expects >= 5
    c_bins, e_bins, ca, ea = [], [], 0.0, 0.0
    for i in order:
        ca += counts[i]
        ea += exp[i]
        if ea >= 5:
            c_bins.append(ca)
            e_bins.append(ea)
            ca = ea = 0.0
    if ea > 0:
        c_bins[-1] += ca
        e_bins[-1] += ea
    c_bins, e_bins = np.array(c_bins), np.array(e_bins)
    chi2 = ((c_bins - e_bins) ** 2 / e_bins).sum()
    return stats.chi2.sf(chi2, len(c_bins) - 1)


@pytest.fixture(scope="module")
def sampling_runs(orc):
    rng = np.random.default_rng(2026)
    L, V, T = 3, 48, 1.0
    Z = (rng.standard_normal((L, V)) * 1.3).astype(np.float32)
    p0 = _softmax(Z[0], T)
    x1 = int(np.argsort(-p0)[1])  # second most likely token: moderate acceptance
    p1 = _softmax(Z[1], T)
    x2 = int(np.argmax(p1))
    path = np.array([x1, x2], np.int32)
    n = 1_000_000
    out, acc = orc.verify_sampling_many(Z, path, T, seed0=777, n=n)
    return dict(Z=Z, T=T, path=path, out=out, acc=acc, n=n, V=V, L=L)


def test_sampling_first_token_marginal_is_target(sampling_runs):
    r = sampling_runs
    counts = np.bincount(r["out"][:, 0], minlength=r["V"]).astype(np.float64)
    assert _chi2_pvalue(counts, _softmax(r["Z"][0], r["T"])) > 0.01


def test_sampling_second_token_conditional_is_target(sampling_runs):
    r = sampling_runs
    kept = r["out"][:, 0] == r["path"][0]
    assert np.all(r["acc"][~kept] == 1)
    counts = np.bincount(r["out"][kept, 1], minlength=r["V"]).astype(np.float64)
    assert counts.sum() > 50_000
    assert _chi2_pvalue(counts, _softmax(r["Z"][1], r["T"])) > 0.01


def test_sampling_bonus_token_after_full_acceptance_is_target(sampling_runs):
    r = sampling_runs
    full = r["acc"] == r["L"]
    counts = np.bincount(r["out"][full, 2], minlength=r["V"]).astype(np.float64)
    assert counts.sum() > 20_000
    assert _chi2_pvalue(counts, _softmax(r["Z"][2], r["T"])) > 0.01


def test_sampling_accept_rate_is_target_probability(sampling_runs):
    r = sampling_runs
    p = _softmax(r["Z"][0], r["T"])[r["path"][0]]
    k = int((r["acc"] >= 2).sum())
    assert stats.binomtest(k, r["n"], p).pvalue > 0.01


def test_sampling_rejection_never_reemits_proposal(sampling_runs):
    r = sampling_runs
    rej1 = r["acc"] == 1
    assert np.all(r["out"][rej1, 0] != r["path"][0])
    rej2 = r["acc"] == 2
    assert np.all(r["out"][rej2, 1] != r["path"][1])


def test_sampling_low_temperature_equals_greedy(orc):
    rng = np.random.default_rng(9)
    for _ in range(20):
        L, V = 6, 100
        Z = rng.permutation(np.arange(L * V, dtype=np.float32)).reshape(L, V) / 10.0  # distinct
        y = np.argmax(Z, 1)
        path = y[:L - 1].copy()
        path[int(rng.integers(0, L - 1))] = 0 if y[0] != 0 else 1
        g_out, g_acc = orc.verify_greedy(Z, path)
        s_out, s_acc, _, _ = orc.verify_sampling(Z, path, T=1e-3, seed=int(rng.integers(1 << 30)))
        assert s_acc == g_acc and s_out.tolist() == g_out.tolist()


def test_sampling_certain_token_always_accepted(orc):
    L, V = 5, 64
    Z = np.zeros((L, V), np.float32)
    path = np.array([3, 9, 27, 40], np.int32)
    for i, x in enumerate(path):
        Z[i, x] = 200.0  # p(x) rounds to 1
    for seed in range(200):
        out, acc, _, _ = orc.verify_sampling(Z, path, T=1.0, seed=seed)
        assert acc == L and out[:L - 1].tolist() == path.tolist()


def test_sampling_depends_on_request_index_and_seed(orc):
    rng = np.random.default_rng(12)
    Z = rng.standard_normal((4, 256)).astype(np.float32)
    path = np.array([1, 2, 3], np.int32)
    a = [tuple(orc.verify_sampling(Z, path, 1.0, seed=5, b=b)[0]) for b in range(50)]
    s = [tuple(orc.verify_sampling(Z, path, 1.0, seed=sd, b=0)[0]) for sd in range(50)]
    assert len(set(a)) > 10 and len(set(s)) > 10
    assert tuple(orc.verify_sampling(Z, path, 1.0, seed=5, b=3)[0].tolist()) == a[3]


@pytest.fixture(scope="module")
def multiblock_runs(orc):
    """A vocabulary of 9192 tokens in three blocks (4096, 4096, 1000) with very different
    masses; the proposal has negligible probability, so every draw is a redraw."""
    rng = np.random.default_rng(99)
    V, T = 2 * 4096 + 1000, 1.0
    z = rng.standard_normal(V)
    z[4096:8192] += 1.0
    z[8192:] += 2.0
    x = 17
    z[x] = -40.0
    Z = np.stack([z, rng.standard_normal(V)]).astype(np.float32)
    n = 120_000
    out, acc = orc.verify_sampling_many(Z, np.array([x], np.int32), T, seed0=31, n=n)
    return dict(Z=Z, T=T, x=x, out=out, acc=acc, n=n, V=V)


def test_redraw_block_masses_follow_residual_target(multiblock_runs):
    r = multiblock_runs
    assert np.all(r["acc"] == 1)
    p = _softmax(r["Z"][0], r["T"])
    p[r["x"]] = 0.0
    p /= p.sum()
    block = r["out"][:, 0] // 4096
    counts = np.bincount(block, minlength=3).astype(np.float64)
    expect = np.array([p[:4096].sum(), p[4096:8192].sum(), p[8192:].sum()])
    assert _chi2_pvalue(counts, expect) > 0.01


def test_redraw_token_distribution_is_residual_target(multiblock_runs):
    r = multiblock_runs
    p = _softmax(r["Z"][0], r["T"])
    p[r["x"]] = 0.0
    p /= p.sum()
    counts = np.bincount(r["out"][:, 0], minlength=r["V"]).astype(np.float64)
    assert counts[r["x"]] == 0
    assert _chi2_pvalue(counts, p) > 0.01


# ------------------------------------------------- the redraw enumerated over uniforms
N_GRID = 1 << 16


def _grid():
    return (np.arange(N_GRID, dtype=np.float64) + 0.5) / N_GRID


def _check_inverse_cdf(tokens, probs):
    """On the grid of N uniforms (j + 1/2) / N, an exact inverse-CDF sampler in vocabulary
    order draws each token a number of times within one of N times its probability (the
    grid points in an interval of length p number N p rounded up or down), and the tokens
    drawn do not decrease as the uniform grows."""
    counts = np.bincount(tokens, minlength=probs.size).astype(np.float64)
    assert counts.sum() == N_GRID
    assert np.all(np.abs(counts - N_GRID * probs) <= 1.0), (counts, N_GRID * probs)
    assert np.all(np.diff(tokens) >= 0)


@pytest.mark.parametrize("V,T,excl", [(9, 0.7, 3), (9, 1.0, -1), (64, 2.5, 0), (64, 0.3, 63)])
def test_redraw_enumerated_is_exact_without_the_rejected_token(orc, V, T, excl):
    """The redraw after a rejected token x draws from softmax(z/T) with x removed and
    renormalised ("DFlash 2: Keep Drafting Parallel", §"A lightweight path selector":
    rejection sampling recovers the exact target distribution); without a rejected token
    (the bonus row), from softmax(z/T) itself."""
    rng = np.random.default_rng(V + excl + 7)
    z = (rng.standard_normal(V) * 2).astype(np.float32)
    p = _softmax(z, T)
    if excl >= 0:
        p[excl] = 0.0
        p /= p.sum()
    tok, _ = orc.redraw_uniforms(z, T, _grid(), excl=excl)
    if excl >= 0:
        assert not np.any(tok == excl)
    _check_inverse_cdf(tok, p)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_redraw_enumerated_residual_of_a_sampled_proposal(orc, seed):
    """The redraw after rejecting a sampled proposal q draws from max(0, p - q)
    renormalised (speculative sampling's residual)."""
    rng = np.random.default_rng(seed)
    V, T, K = 40, 1.3, 6
    z = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = _softmax(z, T)
    cand = rng.choice(V, K, replace=False).astype(np.int32)
    q = rng.dirichlet(np.ones(K))
    r = p.copy()
    r[cand] = np.maximum(0.0, p[cand] - q)
    r /= r.sum()
    tok, _ = orc.redraw_uniforms(z, T, _grid(), cand=cand, q=q)
    _check_inverse_cdf(tok, r)
    # a candidate that the proposal over-weights (q >= p) is never drawn
    assert not np.any(np.isin(tok, cand[q >= p[cand]]))
