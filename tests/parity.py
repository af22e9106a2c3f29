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


# ------------------------------------------------------------------ whole-step comparison
RULES = ("topk", "path", "accept", "draw")


def new_tally() -> dict:
    """Counts of one comparison run: requests compared, requests identical to the oracle,
    the oracle's near-ties per rule (rows for topk, requests otherwise), and the requests
    excluded on each rule because the GPU decided a near-tie differently."""
    return {"requests": 0, "exact": 0, "near": {r: 0 for r in RULES},
            "excluded": {r: 0 for r in RULES}}


def compare_request(g, o, b, q, spec, T, tally) -> bool:
    """Request b of the GPU's fused outputs g against list position q of the oracle's o.

    Ids, paths and accept lengths must be identical, scores within SCORE_RTOL. Where a GPU
    decision differs, the oracle must show a near-tie for that decision; the request is then
    counted under that rule and nothing downstream of the decision is compared. A top-16 set
    that differs at position p leaves positions 1..p-1 compared (their candidates, logits and
    pair scores). Returns whether the request matched exactly."""
    P = spec.L - 1
    tally["requests"] += 1
    ties = [bool(o["topk_gap"][q, p] < TOPK_GAP * abs(o["cand_U"][q, p, -1])) for p in range(P)]
    tally["near"]["topk"] += sum(ties)
    tally["near"]["path"] += int(o["path_margin"][q] < PATH_MARGIN)
    if T > 0:
        tally["near"]["accept"] += int(o["acc_margin"][q] < ACC_MARGIN)
        tally["near"]["draw"] += int(o["draw_margin"][q] < DRAW_MARGIN)
    first = P
    for p in range(P):
        if sorted(g["cand_ids"][b, p].tolist()) != sorted(o["cand_ids"][q, p].tolist()):
            assert ties[p], f"request {b} position {p + 1}: top-16 differs without a near-tie"
            first = p
            break
    for p in range(first):
        gi, gU = g["cand_ids"][b, p], g["cand_U"][b, p]
        pos = {int(t): j for j, t in enumerate(gi)}
        U_in_oracle_order = np.array([gU[pos[int(t)]] for t in o["cand_ids"][q, p]])
        assert np.all(close(U_in_oracle_order, o["cand_U"][q, p])), \
            f"request {b} position {p + 1}: candidate logits"
        assert all(gU[j] > gU[j + 1] or (gU[j] == gU[j + 1] and gi[j] < gi[j + 1])
                   for j in range(15)), f"request {b} position {p + 1}: candidate order"
        Sg = reorder_S_to(o["cand_ids"][q, p - 1] if p else None, o["cand_ids"][q, p],
                          g["cand_ids"][b, p - 1] if p else None, gi, g["S"][b, p], p == 0)
        assert np.all(close(Sg, o["S"][q, p])), f"request {b} position {p + 1}: pair scores"
    if first < P:
        tally["excluded"]["topk"] += 1
        return False
    if g["path"][b].tolist() != o["path"][q].tolist():
        assert o["path_margin"][q] < PATH_MARGIN, f"request {b}: path differs without a near-tie"
        tally["excluded"]["path"] += 1
        return False
    assert close(g["path_score"][b], o["path_score"][q]), f"request {b}: path score"
    if (g["accept_len"][b] != o["accept_len"][q]
            or g["out_tokens"][b].tolist() != o["out_tokens"][q].tolist()):
        assert T > 0 and (o["acc_margin"][q] < ACC_MARGIN or o["draw_margin"][q] < DRAW_MARGIN), \
            f"request {b}: verification differs without a near-tie"
        tally["excluded"]["accept" if o["acc_margin"][q] < ACC_MARGIN else "draw"] += 1
        return False
    tally["exact"] += 1
    return True


def oracle_head(orc, npd, spec, Wq=None, w_scale=None) -> dict:
    """The oracle's LM head, top-16 and gate for every drafted row of a workload, computed
    once (the mode- and temperature-independent part of the step). With Wq / w_scale the
    head is the E4M3 one (rows quantised per row, then the E4M3 product)."""
    B, L = spec.B, spec.L
    P = L - 1
    rows = np.array([b * L + t for b in range(B) for t in range(1, L)])
    if Wq is None:
        u = orc.logits(npd["h"], npd["W"], rows)
    else:
        q, hs = orc.quantize_rows_e4m3(npd["h"], rows)
        u = orc.logits_e4m3(q, hs, Wq, w_scale)
    ids, U, gap = orc.topk(u, 16)
    del u
    g = orc.gate(npd["h"], npd["Wg"], rows)
    return {"cand_ids": ids.reshape(B, P, 16), "cand_U": U.reshape(B, P, 16),
            "topk_gap": gap.reshape(B, P), "gate": g.reshape(B, P, -1)}


def oracle_step(orc, npd, spec, head, mode, T, seed, x0=None, Z=None) -> dict:
    """The oracle's whole step for every request of the workload, composed from its stages
    (pair scores, path, verification) on a precomputed head; the same composition
    orc.select_verify makes (a CPU test pins the two equal). x0 and Z default to the
    workload's."""
    B, P = spec.B, spec.L - 1
    x0 = npd["x0"] if x0 is None else x0
    Z = npd["Z"] if Z is None else Z
    o = {k: head[k] for k in ("cand_ids", "cand_U", "topk_gap")}
    o.update({"S": np.empty((B, P, 16, 16)), "path": np.empty((B, P), np.int32),
              "path_score": np.empty(B), "path_margin": np.empty(B),
              "out_tokens": np.empty((B, spec.L), np.int32), "accept_len": np.empty(B, np.int32),
              "acc_margin": np.full(B, np.inf), "draw_margin": np.full(B, np.inf)})
    sampled = mode in (binding.DFS_PATH_SAMPLE, binding.DFS_PATH_SAMPLE_JOINT) and T > 0
    for b in range(B):
        ids = head["cand_ids"][b]
        S = orc.pair_scores(npd["A"], npd["Bt"], ids, head["cand_U"][b], head["gate"][b], int(x0[b]))
        o["S"][b] = S
        if sampled:
            draw = orc.path_sample_joint if mode == binding.DFS_PATH_SAMPLE_JOINT else orc.path_sample
            path, pidx, q, score, margin = draw(S, ids, T, seed, b)
            out, acc, am, dm = orc.verify_proposal(Z[b], path, ids, q, pidx, T, seed, b)
        else:
            viterbi = mode in (binding.DFS_PATH_VITERBI, binding.DFS_PATH_SAMPLE_JOINT)
            fn = orc.path_viterbi if viterbi else orc.path_greedy
            path, _, score, margin = fn(S, ids)
            if T > 0:
                out, acc, am, dm = orc.verify_sampling(Z[b], path, T, seed, b)
            else:
                (out, acc), am, dm = orc.verify_greedy(Z[b], path), np.inf, np.inf
        o["path"][b], o["path_score"][b], o["path_margin"][b] = path, score, margin
        o["out_tokens"][b], o["accept_len"][b] = out, acc
        o["acc_margin"][b], o["draw_margin"][b] = am, dm
    return o


# near-tie tallies of the GPU comparisons, printed at the end of the session
REPORT: list = []


def report(name: str, tally: dict) -> None:
    REPORT.append((name, tally))
