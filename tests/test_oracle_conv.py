"""Pins for the oracle's two-tap dynamic depthwise convolution (oracle.cpp: orc_conv2tap),
"DFlash 2: Keep Drafting Parallel" §"A lightweight local convolution" (equation and Fig. 4),
checked against what the equation and the stated structure fix rather than against a
retyped formula:

  * zero correction with base kernels (1, 0) is the identity and (0, 1) the shift by one
    position, with nothing before position 0 (block-local, stateless);
  * a correction map with one non-zero entry moves exactly one group of 16 channels of one
    tap, by the position's own input: the group index is c // 16, tap 0 scales x_t and tap 1
    scales x_{t-1}, and the correction is read from row t, not from row t-1;
  * each output depends on its own block and on positions t and t-1 only;
  * the reading's parameter count (a base kernel per tap plus a full linear map to one
    correction per 16 channels and tap) reproduces the 16.5M the page reports for a
    five-layer width-2560 drafter with a convolution before and after each sublayer.
"""
import numpy as np
import pytest

from draft_speculative_decoding_gb300 import workloads as wl


def _bf16(a):
    import torch
    return wl.to_numpy_bits(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def _widen(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _x(B, L, d, seed, bf16=True):
    x = np.random.default_rng(seed).standard_normal((B, L, d)).astype(np.float32)
    return _bf16(x) if bf16 else x


@pytest.mark.parametrize("bf16", [True, False])
def test_identity_and_shift_kernels(orc, bf16):
    B, L, d = 3, 5, 64
    x = _x(B, L, d, 1, bf16)
    xv = _widen(x) if bf16 else x.astype(np.float64)
    Wc = np.zeros((d // 8, d), np.float32)
    ident = orc.conv2tap(x, np.stack([np.ones(d), np.zeros(d)]).astype(np.float32), Wc)
    assert np.array_equal(ident, xv)
    shift = orc.conv2tap(x, np.stack([np.zeros(d), np.ones(d)]).astype(np.float32), Wc)
    assert np.array_equal(shift[:, 1:], xv[:, :-1])
    assert not shift[:, 0].any()  # the verified slot has no predecessor inside the block


@pytest.mark.parametrize("tap,g,k", [(0, 0, 0), (0, 3, 17), (1, 1, 40), (1, 3, 63)])
def test_one_correction_entry_moves_one_group(orc, tap, g, k):
    B, L, d = 2, 4, 64
    G = d // 16
    x = _x(B, L, d, 2, bf16=False)
    Wc = np.zeros((d // 8, d), np.float32)
    Wc[tap * G + g, k] = 1.0  # the correction of (tap, group g) is x_t[k]
    out = orc.conv2tap(x, np.zeros((2, d), np.float32), Wc)
    xv = x.astype(np.float64)
    group = np.zeros(d, bool)
    group[16 * g:16 * g + 16] = True
    assert not out[:, :, ~group].any()
    for t in range(L):
        src = xv[:, t] if tap == 0 else (xv[:, t - 1] if t > 0 else np.zeros_like(xv[:, t]))
        want = xv[:, t, k][:, None] * src[:, group]  # scaled by row t's own channel k
        assert np.array_equal(out[:, t][:, group], want)


def test_locality_and_block_independence(orc):
    B, L, d = 3, 6, 128
    rng = np.random.default_rng(3)
    x = rng.standard_normal((B, L, d)).astype(np.float32)
    base = rng.standard_normal((2, d)).astype(np.float32)
    Wc = (rng.standard_normal((d // 8, d)) * 0.05).astype(np.float32)
    out = orc.conv2tap(x, base, Wc)
    t = 3
    y = x.copy()
    y[:, t + 1] += 1.0
    y[:, t - 2] -= 2.0
    y[1] *= 3.0  # another block entirely
    out2 = orc.conv2tap(y, base, Wc)
    # positions t (reads t, t-1) and t-3 (reads t-3, t-4) are untouched; t-2 and t-1 move
    assert np.array_equal(out2[[0, 2], t], out[[0, 2], t])
    assert np.array_equal(out2[[0, 2], t - 3], out[[0, 2], t - 3])
    assert not np.array_equal(out2[[0, 2], t - 1], out[[0, 2], t - 1])
    perm = [2, 0, 1]
    assert np.array_equal(orc.conv2tap(x[perm], base, Wc), out[perm])


def test_parameter_count_of_the_reading_matches_the_page():
    d, layers, per_layer = 2560, 5, 4  # before and after attention and MLP
    per_conv = 2 * d + 2 * (d // 16) * d  # base kernels + the correction map Wc [d/8, d]
    total = layers * per_layer * per_conv
    assert abs(total - 16.5e6) / 16.5e6 < 0.005  # the page: 16.5M parameters (3 %)
