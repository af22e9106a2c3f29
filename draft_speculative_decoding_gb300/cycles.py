"""Multi-cycle draft-verify loop through the C ABI ("DFlash 2: Keep Drafting Parallel",
Fig. 1 and Table 1: one draft-verify cycle after another, each cycle's last emitted token the
next cycle's last verified token).

fused_cycles: per cycle dfs_select_verify then dfs_next_tokens, the last verified tokens
carried on the device (recordable into one CUDA graph: nothing here synchronises).
"""
from __future__ import annotations

from . import binding


def fused_cycles(dims, data, hs, Zs, x0, ws, mode, n_cycles, seed0=0, outputs=None, stream=None,
                 temperature=0.0, want_intermediates=False):
    """n_cycles fused steps over the rotating inputs hs[c % n], Zs[c % n], cycle c with seed
    seed0 + c; x0 (int32 [B], on the device) is updated in place after every cycle. Returns
    the outputs of the last cycle (path, out_tokens, accept_len, and with want_intermediates
    its candidates and scores) and, per cycle, its accept lengths (device tensors)."""
    accs = []
    for c in range(n_cycles):
        res = binding.dfs_select_verify(dims, hs[c % len(hs)], data["W"], data["Wg"], data["A"],
                                        data["Bt"], x0, Zs[c % len(Zs)], mode, temperature,
                                        seed0 + c, ws, outputs=outputs, stream=stream,
                                        want_intermediates=want_intermediates)
        binding.dfs_next_tokens(res["out_tokens"], res["accept_len"], x0, stream=stream)
        accs.append(res["accept_len"] if outputs is not None else res["accept_len"].clone())
    return res, accs
