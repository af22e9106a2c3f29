"""Pins for the E4M3 LM head of the oracle (orc_e4m3_*, orc_quantize_rows_e4m3,
orc_logits_e4m3), against what the format's definition and the arithmetic fix:

  * decoding all 256 bytes and rounding to nearest even agree with torch's independent
    float8_e4m3fn implementation of the OCP format (including exact ties);
  * the row scale is the smallest power of two that brings the row's largest magnitude
    to at most 448 (closed form: the scaled maximum lies in (224, 448]);
  * quantisation error is at most half a grid step; logits equal a float64 matmul of the
    dequantised operands.
"""
import numpy as np
import pytest
import torch


def test_decode_table_matches_the_format(orc):
    b = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.tolist() == np.isnan(ours).tolist() and nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[~nan].max() == 448.0 and ours[1] == 2.0 ** -9


def test_rounding_to_nearest_even_including_ties(orc):
    grid = np.unique(np.abs(orc.e4m3_decode(np.arange(256, dtype=np.uint8))))
    grid = grid[np.isfinite(grid)]
    mids = (grid[:-1] + grid[1:]) / 2  # exact ties between neighbours
    rng = np.random.default_rng(0)
    x = np.concatenate([grid, mids, -mids, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(20000) * 0.01]).astype(np.float32)
    ours = orc.e4m3_encode(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("scale_pow", [-30, -5, 0, 7])
def test_row_scale_closed_form_and_error_bound(orc, scale_pow):
    rng = np.random.default_rng(scale_pow + 40)
    h = (rng.standard_normal((6, 256)) * 2.0 ** scale_pow).astype(np.float32)
    h[3, :] = 0.0  # an all-zero row: scale 1
    h[4, 7] = np.float32(448.0 * 2.0 ** scale_pow)  # the boundary: scale 2^scale_pow exactly
    h[4, 8:] = 0.0
    q, s = orc.quantize_rows_e4m3(h, np.arange(6))
    assert s[4] == 2.0 ** scale_pow
    amax = np.abs(h).max(axis=1).astype(np.float64)
    for i in range(6):
        assert np.log2(s[i]) == np.round(np.log2(s[i]))  # a power of two
        if amax[i] == 0:
            assert s[i] == 1.0 and not q[i].any()
            continue
        assert 224.0 < amax[i] / s[i] <= 448.0
    deq = orc.e4m3_decode(q.reshape(-1)).reshape(q.shape) * s[:, None]
    x = h.astype(np.float64) / s[:, None]
    # grid step at |x|: 2^(floor(log2|x|) - 3) for |x| >= 2^-6, else 2^-9
    step = np.where(np.abs(x) >= 2.0 ** -6,
                    2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -6))) - 3), 2.0 ** -9)
    assert np.all(np.abs(deq / s[:, None] - x) <= step / 2)


def test_e4m3_logits_are_the_dequantised_product(orc):
    rng = np.random.default_rng(5)
    n, d, V = 5, 192, 300
    q = rng.integers(0, 256, (n, d), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0  # no NaN codes
    Wq = rng.integers(0, 256, (V, d), dtype=np.uint8)
    Wq[(Wq & 0x7F) == 0x7F] = 1
    hs = 2.0 ** rng.integers(-8, 3, n).astype(np.float64)
    ws = (2.0 ** rng.integers(-12, -4, V)).astype(np.float32)
    u = orc.logits_e4m3(q, hs, Wq, ws)
    hd = orc.e4m3_decode(q.reshape(-1)).reshape(n, d) * hs[:, None]
    wd = orc.e4m3_decode(Wq.reshape(-1)).reshape(V, d) * ws[:, None].astype(np.float64)
    assert np.allclose(u, hd @ wd.T, rtol=1e-12, atol=1e-12)


def test_whole_step_with_the_e4m3_head_composes(orc):
    from draft_speculative_decoding_gb300 import workloads as wl
    spec = wl.TINY.with_(name="q", dtype="bf16", B=2, L=4, V=600, d=128, r=16, seed=6,
                         lmhead="e4m3")
    data = wl.generate(spec, "cpu")
    npd = {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}
    Wq, ws = data["Wq"].numpy(), data["w_scale"].numpy()
    res = orc.select_verify(*[npd[k] for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")],
                            Wq=Wq, w_scale=ws)
    rows = np.array([b * spec.L + t for b in range(spec.B) for t in range(1, spec.L)])
    q, s = orc.quantize_rows_e4m3(npd["h"], rows)
    ids, U, _ = orc.topk(orc.logits_e4m3(q, s, Wq, ws), 16)
    assert np.array_equal(res["cand_ids"].reshape(-1, 16), ids)
    assert np.array_equal(res["cand_U"].reshape(-1, 16), U)
