"""Checks of the multi-cycle loop against targets planted by the test itself (shared by
the GPU tests and the benchmark's planted leg; none of this is library code).

* plant_target_argmax: a synthetic target whose argmax agrees with each drafted token with a
  given per-position probability, independently, so the accept length of greedy
  verification has the closed form 1 + sum_k prod_{i<=k} r_i ("DFlash 2: Keep Drafting
  Parallel", Table 1: 4.27 for its Recall@1 row).
* planted_cycles: staged greedy cycles (dfs_lmhead_topk, dfs_pair_score, dfs_path_select,
  then the planted target, dfs_verify and the hand-off).
* leading_agreements and closed_form_accept_len: what the accept lengths must be.
"""
from __future__ import annotations

import torch

from draft_speculative_decoding_gb300 import binding

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


def plant_target_argmax(Z: torch.Tensor, path: torch.Tensor, recall, gen: torch.Generator):
    """Synthetic target for a decode loop: in place, each target row i of Z [B, L, V] gets a
    planted argmax (logit 64, above any drawn value) that equals the drafted token path[:, i]
    with probability recall[i], independently per row and request, and otherwise another
    token drawn uniformly; the bonus row L-1 gets a uniform token. Returns (agree [B, L-1]
    bool, handle) where handle restores Z with restore_target(Z, handle)."""
    B, L, V = Z.shape
    dev = Z.device
    r = torch.as_tensor(list(recall)[:L - 1], dtype=torch.float32, device=dev)
    agree = torch.rand(B, L - 1, generator=gen, device=dev) < r[None, :]
    other = (path.long() + 1 + torch.randint(0, V - 1, (B, L - 1), generator=gen, device=dev)) % V
    tok = torch.cat([torch.where(agree, path.long(), other),
                     torch.randint(0, V, (B, 1), generator=gen, device=dev)], dim=1)
    bi = torch.arange(B, device=dev)[:, None].expand(B, L)
    ti = torch.arange(L, device=dev)[None, :].expand(B, L)
    saved = Z[bi, ti, tok].clone()
    Z[bi, ti, tok] = 64.0
    return agree, (bi, ti, tok, saved)


def restore_target(Z: torch.Tensor, handle) -> None:
    bi, ti, tok, saved = handle
    Z[bi, ti, tok] = saved


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
        agree, handle = plant_target_argmax(Z, path, recall, gen)
        toks, acc = binding.dfs_verify(dims, path, Z, 0.0, c, ws, stream=stream)
        restore_target(Z, handle)
        binding.dfs_next_tokens(toks, acc, x0, stream=stream)
        out.append((acc, agree))
    return out


def leading_agreements(agree: torch.Tensor) -> torch.Tensor:
    """1 + the number of leading True per row of agree [B, P]: the accept length greedy
    verification must report against a planted target."""
    return 1 + torch.cumprod(agree.int(), dim=1).sum(dim=1)
