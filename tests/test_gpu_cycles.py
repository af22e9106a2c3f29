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

import pytest
import torch

from draft_speculative_decoding_gb300 import binding, cycles
from draft_speculative_decoding_gb300 import workloads as wl
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
    runs = cycles.planted_cycles(dims, data, [data["h"]], data["Z"], x0, ws, recall, 60, gen)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    accs = torch.stack([a for a, _ in runs])
    for acc, agree in runs:
        assert torch.equal(acc.long(), cycles.leading_agreements(agree))
    n = accs.numel()
    mean, sd = accs.float().mean().item(), accs.float().std().item()
    want = cycles.closed_form_accept_len(recall)
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
