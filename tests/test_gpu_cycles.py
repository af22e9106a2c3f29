"""The multi-cycle draft-verify loop on the GPU (cycles.py through the C ABI):

  * against targets planted to agree with each drafted token with the page's Table 1 Recall@1
    probabilities, every cycle's accept length equals 1 + the leading run of agreements
    (exact), and the mean over cycles and requests matches the closed form 4.27 within its
    statistical error ("DFlash 2: Keep Drafting Parallel", Table 1);
  * dfs_next_tokens hands each request's last emitted token to the next cycle, and a fused
    loop recorded into a CUDA graph replays the eager loop bit for bit."""
import json
import math
import os

import numpy as np

import pytest
import torch

from draft_speculative_decoding_gb300 import binding, cycles
from draft_speculative_decoding_gb300 import workloads as wl
import planted
from parity import dims_for

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "blog_table1_recall.json")
SPEC = wl.TINY.with_(name="cycles", dtype="bf16", B=32, L=8, V=4096, d=256, r=64, seed=71)


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def test_planted_cycles_accept_lengths(lib):
    data = wl.generate(SPEC, "cuda")
    dims = dims_for(SPEC)
    ws = binding.alloc_workspace(dims)
    recall = json.load(open(GOLDEN))["recall_at_1"]
    x0 = data["x0"].clone()
    gen = torch.Generator(device="cuda").manual_seed(5)
    runs = planted.planted_cycles(dims, data, [data["h"]], data["Z"], x0, ws, recall, 60, gen)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    accs = torch.stack([a for a, _ in runs])
    for acc, agree in runs:
        assert torch.equal(acc.long(), planted.leading_agreements(agree))
    n = accs.numel()
    mean, sd = accs.float().mean().item(), accs.float().std().item()
    want = planted.closed_form_accept_len(recall)
    assert abs(mean - want) < 4 * sd / math.sqrt(n), (mean, want)


def test_next_tokens_hand_off_and_bounds(lib):
    out = torch.arange(3 * 4, dtype=torch.int32, device="cuda").view(3, 4)
    acc = torch.tensor([1, 4, 0], dtype=torch.int32, device="cuda")
    nxt = binding.dfs_next_tokens(out, acc)
    assert nxt.tolist() == [0, 7, -1]


def test_fused_loop_hands_off_and_replays_from_a_graph(lib):
    spec = SPEC.with_(B=8, seed=72)
    data = wl.generate(spec, "cuda")
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    hs, Zs = [data["h"]], [data["Z"], wl.fresh_targets(data, 9)]
    P = spec.L - 1

    def outs():
        return (torch.zeros(spec.B, P, dtype=torch.int32, device="cuda"),
                torch.zeros(spec.B, spec.L, dtype=torch.int32, device="cuda"),
                torch.zeros(spec.B, dtype=torch.int32, device="cuda"))

    # eager, cycle by cycle, checking the hand-off
    x0 = data["x0"].clone()
    for c in range(4):
        res, _ = cycles.fused_cycles(dims, data, hs, Zs[c % 2:] + Zs[:c % 2], x0, ws,
                                     binding.DFS_PATH_GREEDY, 1, seed0=c)
        o, a = res["out_tokens"], res["accept_len"]
        last = o.gather(1, (a.long() - 1)[:, None])[:, 0]
        assert torch.equal(x0, last)
    eager_x0 = x0.clone()
    # the same four cycles recorded into one graph
    o3 = outs()
    x0g = data["x0"].clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cycles.fused_cycles(dims, data, hs, Zs, x0g, ws, binding.DFS_PATH_GREEDY, 4, outputs=o3)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    x0g.copy_(data["x0"])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cycles.fused_cycles(dims, data, hs, Zs, x0g, ws, binding.DFS_PATH_GREEDY, 4, outputs=o3)
    x0g.copy_(data["x0"])
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(x0g, eager_x0)
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK


@pytest.mark.parametrize("mode,T", [(binding.DFS_PATH_GREEDY, 0.0), (binding.DFS_PATH_VITERBI, 0.8),
                                    (binding.DFS_PATH_SAMPLE, 0.8)])
def test_fused_loop_matches_the_oracle_cycle_by_cycle(lib, orc, mode, T):
    """The multi-cycle loop ([Blog] Fig. 1: each cycle's last emitted token is the next
    cycle's last verified token) against the oracle run the same way: five cycles at B = 8
    over rotating hidden states and target logits, the oracle's x0 handed off from its own
    outputs. Every cycle's path, tokens and accept length must be identical; a request that
    diverges on a near-tie is counted and dropped from the later cycles (its x0 differs)."""
    from parity import compare_request, new_tally, np_inputs, oracle_head, oracle_step, report
    spec = SPEC.with_(name="cycles_oracle", B=8, seed=73)
    data = wl.generate(spec, "cuda")
    hs = [data["h"], data["h"].roll(1, dims=0).contiguous()]
    Zs = [data["Z"], wl.fresh_targets(data, 31), wl.fresh_targets(data, 32)]
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    npd = np_inputs(data)
    heads = []
    for h in hs:  # the oracle's LM head of each hidden-state set, once
        npd_h = dict(npd, h=wl.to_numpy_bits(h))
        heads.append((npd_h, oracle_head(orc, npd_h, spec)))
    x0 = data["x0"].clone()
    x0_o = npd["x0"].copy()
    live = set(range(spec.B))
    tally = new_tally()
    n_cycles = 5
    for c in range(n_cycles):
        res, _ = cycles.fused_cycles(dims, data, [hs[c % 2]], [Zs[c % 3]], x0, ws, mode, 1,
                                     seed0=100 + c, temperature=T, want_intermediates=True)
        torch.cuda.synchronize()
        assert binding.dfs_get_device_error(ws) == binding.DFS_OK
        g = {k: v.cpu().numpy() for k, v in res.items()}
        npd_h, head = heads[c % 2]
        o = oracle_step(orc, npd_h, spec, head, mode, T, 100 + c, x0=x0_o,
                        Z=wl.to_numpy_bits(Zs[c % 3]))
        for b in sorted(live):
            if not compare_request(g, o, b, b, spec, T, tally):
                live.discard(b)
        # the oracle's own hand-off: each request's last emitted token
        x0_o = np.array([o["out_tokens"][b][o["accept_len"][b] - 1] for b in range(spec.B)],
                        np.int32)
        # the loop's hand-off on the device equals the oracle's for every request still live
        got = x0.cpu().numpy()
        assert all(got[b] == x0_o[b] for b in live), f"cycle {c}: hand-off differs"
    report(f"{spec.name} mode={mode} T={T} ({n_cycles} cycles)", tally)
    assert len(live) >= spec.B - 2
