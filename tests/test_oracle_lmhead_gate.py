"""Pins for the oracle's LM-head logits, keep-top-K and context gate.

Logits and top-K are pinned to numpy's float64 matmul and lexsort on the same
bytes. The gate's form is a reading, so it is pinned by closed-form special
cases that any indexing, transposition or sign slip breaks."""
import numpy as np
import pytest


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _widen_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("V,d,n", [(1000, 64, 3), (5003, 192, 5)])
def test_logits_match_numpy_float64(orc, dtype, V, d, n):
    rng = np.random.default_rng(V + d)
    h = rng.standard_normal((n + 2, d)).astype(np.float32)
    W = (rng.standard_normal((d, V)) / np.sqrt(d)).astype(np.float32)
    if dtype == "bf16":
        h, W = _bf16_bits(h), _bf16_bits(W)
        hd, Wd = _widen_bits(h), _widen_bits(W)
    else:
        hd, Wd = h.astype(np.float64), W.astype(np.float64)
    rows = np.array([1, 0, n + 1, 2, 3][:n], np.int64)
    u = orc.logits(h, W, rows, nthreads=3)
    ref = hd[rows] @ Wd
    np.testing.assert_allclose(u, ref, rtol=1e-12, atol=1e-12)


def test_topk_matches_lexsort_with_planted_ties(orc):
    rng = np.random.default_rng(7)
    n, V, K = 6, 777, 16
    u = rng.standard_normal((n, V))
    # plant exact ties inside the top and exactly at the K/K+1 boundary
    order = np.argsort(-u[0], kind="stable")
    u[0, order[3]] = u[0, order[2]]
    u[1, 5] = u[1, 700] = u[1].max() + 1.0
    o2 = np.argsort(-u[2], kind="stable")
    u[2, o2[16]] = u[2, o2[15]]
    ids, U, gap = orc.topk(u, K)
    for i in range(n):
        ref = np.lexsort((np.arange(V), -u[i]))[:K]
        assert ids[i].tolist() == ref.tolist()
        np.testing.assert_array_equal(U[i], u[i, ref])
        srt = np.sort(u[i])[::-1]
        assert gap[i] == srt[K - 1] - srt[K]
    assert ids[1, 0] == 5 and ids[1, 1] == 700
    assert gap[2] == 0.0


def test_topk_rejects_short_vocab(orc):
    with pytest.raises(ValueError):
        orc.topk(np.zeros((1, 8)), 16)


def test_gate_zero_weights_give_one_half(orc):
    h = np.random.default_rng(0).standard_normal((4, 32)).astype(np.float32)
    Wg = np.zeros((8, 32), np.float32)
    g = orc.gate(h, Wg, [0, 3])
    assert np.all(g == 0.5)


def test_gate_one_hot_weight_picks_row_and_column(orc):
    # Wg[j0, k0] = w; h row with h[k0] = x: only gate j0 moves, to sigmoid(w*x)
    r, d = 6, 20
    j0, k0, w, x = 4, 13, 0.75, -2.0
    Wg = np.zeros((r, d), np.float32)
    Wg[j0, k0] = w
    h = np.zeros((3, d), np.float32)
    h[2, k0] = x
    h[1, j0] = 5.0  # a transposed read (Wg[k][j] or h[j]) would pick this up
    g = orc.gate(h, Wg, [2, 1])
    expect = np.full((2, r), 0.5)
    expect[0, j0] = 1.0 / (1.0 + np.exp(-(w * x)))
    np.testing.assert_allclose(g, expect, rtol=0, atol=1e-15)


def test_gate_sign_flip_is_complement(orc):
    rng = np.random.default_rng(3)
    h = rng.standard_normal((5, 48)).astype(np.float32)
    Wg = rng.standard_normal((16, 48)).astype(np.float32) / 7
    g = orc.gate(h, Wg, [0, 1, 4])
    gneg = orc.gate(h, -Wg, [0, 1, 4])
    np.testing.assert_allclose(g + gneg, 1.0, rtol=0, atol=1e-14)
    assert np.all((g > 0) & (g < 1))
