"""Host logic of the planted-target checks of the multi-cycle loop (tests/planted.py), on the
CPU:

  * the accept-length closed form reproduces the verify lengths the page prints for its
    Table 1 rows ("DFlash 2: Keep Drafting Parallel", §"The right tokens are already there"),
    from the golden file's recall rows;
  * the planted target's argmax is the drafted token exactly where `agree` says so, and
    restoring gives back the original bytes;
  * the accept length implied by the planted agreements is 1 + the leading run of agreements.
"""
import json
import os

import pytest
import torch

import planted

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "blog_table1_recall.json")


def test_closed_form_reproduces_table1_verify_lengths():
    g = json.load(open(GOLDEN))
    tol = g["printed_precision"]
    assert abs(planted.closed_form_accept_len(g["recall_at_1"]) - g["verify_length_recall_at_1"]) <= tol
    assert abs(planted.closed_form_accept_len(g["recall_at_16"]) - g["verify_length_recall_at_16"]) <= tol
    assert planted.closed_form_accept_len([]) == 1.0
    assert planted.closed_form_accept_len([1.0] * 7) == 8.0
    assert planted.closed_form_accept_len([0.0, 1.0, 1.0]) == 1.0
    assert list(planted.TABLE1_RECALL_AT_1) == g["recall_at_1"]


def test_planted_target_argmax_and_restore():
    B, L, V = 6, 8, 300
    gen = torch.Generator().manual_seed(3)
    Z = torch.randn(B, L, V, generator=gen).to(torch.bfloat16)
    Z0 = Z.clone()
    path = torch.randint(0, V, (B, L - 1), generator=gen, dtype=torch.int32)
    agree, handle = planted.plant_target_argmax(Z, path, [0.5] * 7, gen)
    am = Z.float().argmax(dim=2)
    assert torch.equal(am[:, :-1] == path.long(), agree)
    assert 0 < agree.sum() < agree.numel()
    planted.restore_target(Z, handle)
    assert torch.equal(Z.view(torch.int16), Z0.view(torch.int16))


@pytest.mark.parametrize("row,want", [([1, 1, 0, 1], 3), ([0, 1, 1, 1], 1), ([1, 1, 1, 1], 5),
                                      ([0, 0, 0, 0], 1)])
def test_leading_agreements(row, want):
    assert planted.leading_agreements(torch.tensor([row], dtype=torch.bool)).item() == want
