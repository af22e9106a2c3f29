"""Multi-cycle draft-verify loops through the C ABI ("DFlash 2: Keep Drafting Parallel",
Fig. 1 and Table 1: one draft-verify cycle after another, each cycle's last emitted token the
next cycle's last verified token).

* fused_cycles: per cycle dfs_select_verify then dfs_next_tokens, the last verified tokens
  carried on the device (recordable into one CUDA graph: nothing here synchronises).
* planted_cycles: per cycle the stages (dfs_lmhead_topk, dfs_pair_score, dfs_path_select),
  then a synthetic target whose argmax agrees with each drafted token with a given
  per-position probability (workloads.plant_target_argmax), then dfs_verify and the hand-off.
  With independent agreements the mean accept length has the closed form
  1 + sum_k prod_{i<=k} r_i ([Blog] Table 1: 4.27 for its Recall@1 row).
"""
from __future__ import annotations

import torch

from . import binding
from . import workloads as wl


# [Blog] Table 1: Recall@1 per draft position (each conditioned on every earlier position being
# correct) of a five-layer Qwen3-4B DFlash on GSM8K; its verify length is 4.27.
TABLE1_RECALL_AT_1 = (0.854, 0.803, 0.794, 0.783, 0.775, 0.759, 0.729)


def closed_form_accept_len(recall) -> float:
    """Expected accept length when draft i is accepted with probability r_i given that every
    earlier draft was (the verify length counts the target's own next token)."""
    total, run = 1.0, 1.0
    for r in recall:
        run *= float(r)
        total += run
    return total


def fused_cycles(dims, data, hs, Zs, x0, ws, mode, n_cycles, seed0=0, outputs=None, stream=None):
    """n_cycles fused steps over the rotating inputs hs[c % n], Zs[c % n]; x0 (int32 [B], on
    the device) is updated in place after every cycle. Returns the outputs of the last cycle
    (path, out_tokens, accept_len) and, per cycle, its accept lengths (device tensors)."""
    accs = []
    for c in range(n_cycles):
        res = binding.dfs_select_verify(dims, hs[c % len(hs)], data["W"], data["Wg"], data["A"],
                                        data["Bt"], x0, Zs[c % len(Zs)], mode, 0.0, seed0 + c,
                                        ws, outputs=outputs, stream=stream)
        binding.dfs_next_tokens(res["out_tokens"], res["accept_len"], x0, stream=stream)
        accs.append(res["accept_len"] if outputs is not None else res["accept_len"].clone())
    return res, accs


def planted_cycles(dims, data, hs, Z, x0, ws, recall, n_cycles, gen, stream=None):
    """n_cycles staged greedy cycles against targets planted in Z (restored after each cycle).
    Returns per cycle (accept_len [B], agree [B, L-1]) as device tensors."""
    out = []
    for c in range(n_cycles):
        h = hs[c % len(hs)]
        ids, U = binding.dfs_lmhead_topk(dims, h, data["W"], ws, stream=stream)
        S = binding.dfs_pair_score(dims, h, data["Wg"], data["A"], data["Bt"], x0, ids, U, ws,
                                   stream=stream)
        path, _ = binding.dfs_path_select(dims, S, ids, binding.DFS_PATH_GREEDY, stream=stream)
        agree, handle = wl.plant_target_argmax(Z, path, recall, gen)
        toks, acc = binding.dfs_verify(dims, path, Z, 0.0, c, ws, stream=stream)
        wl.restore_target(Z, handle)
        binding.dfs_next_tokens(toks, acc, x0, stream=stream)
        out.append((acc, agree))
    return out


def leading_agreements(agree: torch.Tensor) -> torch.Tensor:
    """1 + the number of leading True per row of agree [B, P]: the accept length greedy
    verification must report against a planted target."""
    return 1 + torch.cumprod(agree.int(), dim=1).sum(dim=1)
