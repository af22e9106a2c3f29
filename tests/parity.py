"""Shared helpers for the GPU parity tests: tolerances, near-tie exclusion rules, and the
conversions between the CUDA path's torch tensors and the oracle's numpy inputs.

Rules (where fp32 on the GPU and fp64 in the oracle may legitimately decide differently,
the case is excluded from the exact comparison and counted):
  * scores (U, S, path score) agree within SCORE_RTOL * max(1, |oracle value|);
  * a GPU decision that differs from the oracle's is accepted only where the oracle shows
    a near-tie for that decision, and the case is counted and left out of the comparisons
    downstream of it:
      - top-16 set of a row: boundary gap u_16 - u_17 < TOPK_GAP * |u_16|;
      - path: smallest relative best-vs-second margin on the path < PATH_MARGIN;
      - sampling: an accept test with |U - p| / p < ACC_MARGIN, or a redraw whose target
        lies within DRAW_MARGIN (relative to the row's total) of a cumulative boundary;
  * everywhere else token ids, paths and accept lengths must be identical.
"""
from __future__ import annotations

import numpy as np
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl

SCORE_RTOL = 1e-3
TOPK_GAP = 1e-3
PATH_MARGIN = 1e-3
ACC_MARGIN = 1e-4
DRAW_MARGIN = 1e-4
GATE_ATOL = 1e-4


def np_inputs(data: dict) -> dict:
    return {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}


def dims_for(spec: wl.WorkloadSpec) -> binding.Dims:
    code = binding.DFS_BF16 if spec.dtype == "bf16" else binding.DFS_FP32
    return binding.make_dims(spec.B, spec.L, spec.V, spec.d, spec.r, code, code)


def close(gpu, ref, rtol=SCORE_RTOL):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(gpu - ref) <= rtol * np.maximum(1.0, np.abs(ref))


def topk_near_tie(U_ref_row, gap):
    return gap < TOPK_GAP * abs(U_ref_row[-1])


def compare_topk(g_ids, g_U, o_ids, o_U, o_gap):
    """Per row: the GPU's 16-token set equals the oracle's, with matching logits, in
    (value desc, id asc) order of the GPU's own values. A row whose set differs is allowed
    only when the oracle has a near-tie at the 16/17 boundary; such rows are counted.
    Returns (rows, near-tie rows, rows that diverged on a near-tie)."""
    g_ids = np.asarray(g_ids).reshape(-1, 16)
    g_U = np.asarray(g_U).reshape(-1, 16)
    o_ids = np.asarray(o_ids).reshape(-1, 16)
    o_U = np.asarray(o_U).reshape(-1, 16)
    o_gap = np.asarray(o_gap).reshape(-1)
    near = diverged = 0
    for i in range(o_ids.shape[0]):
        tie = topk_near_tie(o_U[i], o_gap[i])
        near += tie
        if sorted(g_ids[i].tolist()) != sorted(o_ids[i].tolist()):
            assert tie, f"row {i}: top-16 sets differ without a near-tie in the oracle"
            diverged += 1
            continue
        pos = {int(t): j for j, t in enumerate(g_ids[i])}
        gU = np.array([g_U[i, pos[int(t)]] for t in o_ids[i]])
        assert np.all(close(gU, o_U[i])), f"row {i}: logits differ {gU} vs {o_U[i]}"
        for j in range(15):
            a, b = (g_U[i, j], g_ids[i, j]), (g_U[i, j + 1], g_ids[i, j + 1])
            assert a[0] > b[0] or (a[0] == b[0] and a[1] < b[1]), f"row {i}: not ordered"
    return o_ids.shape[0], near, diverged


def reorder_S_to(o_prev_ids, o_cur_ids, g_prev_ids, g_cur_ids, g_S_pos, first: bool):
    """Reindex one position's GPU pair-score matrix into the oracle's candidate order."""
    pc = {int(t): j for j, t in enumerate(g_cur_ids)}
    cols = [pc[int(t)] for t in o_cur_ids]
    if first:
        return g_S_pos[:, cols]
    pp = {int(t): j for j, t in enumerate(g_prev_ids)}
    rows = [pp[int(t)] for t in o_prev_ids]
    return g_S_pos[np.ix_(rows, cols)]


def to_cpu(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()
