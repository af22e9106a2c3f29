"""GPU parity of the fused dfs_select_verify against the oracle's whole step, on every
request: small shapes, and the pages-shaped workloads at full size in the launch
configuration the benchmark times (there the oracle's fp64 LM head is computed once per
workload and the rest of its step once per path mode and temperature). Near-tie exclusions
are counted per workload and rule and printed at the end of the run."""
import numpy as np
import pytest
import torch

from draft_speculative_decoding_gb300 import binding
from draft_speculative_decoding_gb300 import workloads as wl
from parity import (compare_request, dims_for, new_tally, np_inputs, oracle_head, oracle_step,
                    report, to_cpu)

pytestmark = pytest.mark.gpu

SMALL = [
    wl.TINY,
    wl.TINY.with_(name="fused_mt1", dtype="bf16", B=4, L=6, V=6000, d=256, r=64, seed=31),
    wl.TINY.with_(name="fused_mt2", dtype="bf16", B=24, L=8, V=4000, d=320, r=256, seed=32,
                  zipf=True),
    wl.TINY.with_(name="fused_groups", dtype="bf16", B=33, L=9, V=2600, d=128, r=64, seed=33),
    wl.TINY.with_(name="fused_L16", dtype="bf16", B=6, L=16, V=8192, d=192, r=32, seed=34,
                  agreement=("top1_linear", 0.95, 0.6)),
    # CTA-pair LM head at its edges: one row past a single M tile; exactly 256 rows with two
    # gate tiles (r = 512) placed among the first round; fewer vocabulary tiles than pairs
    wl.TINY.with_(name="pairs_129rows", dtype="bf16", B=43, L=3, V=3000, d=128, r=64, seed=35),
    wl.TINY.with_(name="pairs_256rows_r512", dtype="bf16", B=32, L=8, V=5000, d=192, r=512,
                  seed=36, zipf=True),
    wl.TINY.with_(name="pairs_few_tiles", dtype="bf16", B=20, L=8, V=1040, d=64, r=256, seed=37),
    wl.TINY.with_(name="pairs_L16", dtype="bf16", B=16, L=16, V=6000, d=256, r=256, seed=38,
                  agreement=("top1_linear", 0.85, 0.55)),
    # the vocabulary-major LM head, chosen because it saves a pass over W: 288 rows of which
    # 256 drafted (with a gate tile); 320 rows of blocks of 5, 256 drafted
    wl.TINY.with_(name="vt_32x9", dtype="bf16", B=32, L=9, V=3000, d=128, r=256, seed=39,
                  zipf=True),
    wl.TINY.with_(name="vt_64x5", dtype="bf16", B=64, L=5, V=2600, d=128, r=64, seed=40),
    # one draft position (every tail block merges one set; a one-step walk); and a rank that
    # is not a multiple of 16, so the tail's pair scores take the SIMT path on bf16 tables
    wl.TINY.with_(name="fused_L2", dtype="bf16", B=8, L=2, V=3000, d=128, r=32, seed=41),
    wl.TINY.with_(name="fused_r24", dtype="bf16", B=6, L=5, V=2600, d=128, r=24, seed=42),
]


@pytest.fixture(scope="module")
def lib():
    from draft_speculative_decoding_gb300 import build
    build.build()
    return binding.load()


def _run(data, spec, mode, T, seed):
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    res = binding.dfs_select_verify(dims, data["h"], data["W"], data["Wg"], data["A"], data["Bt"],
                                    data["x0"], data["Z"], mode, T, seed, ws,
                                    want_intermediates=True)
    torch.cuda.synchronize()
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    return {k: to_cpu(v) for k, v in res.items()}


def _compare(g, o, spec, reqs, T, name=None):
    """Every listed request compared (parity.compare_request); returns the number excluded on
    a near-tie, and reports the tally under `name` when given."""
    tally = new_tally()
    for q, b in enumerate(reqs):
        compare_request(g, o, b, q, spec, T, tally)
    if name is not None:
        report(name, tally)
    return tally["requests"] - tally["exact"]


def _invariants(g, spec, npd, T):
    """Properties of every request at any size."""
    L, V = spec.L, spec.V
    acc = g["accept_len"]
    assert np.all((acc >= 1) & (acc <= L))
    for b in range(spec.B):
        n = acc[b]
        out = g["out_tokens"][b]
        assert np.all(out[n:] == -1) and np.all((out[:n] >= 0) & (out[:n] < V))
        assert out[:n - 1].tolist() == g["path"][b, :n - 1].tolist()  # accepted drafts are the path
        for p in range(L - 1):  # the path is drawn from each position's candidates
            assert g["path"][b, p] in g["cand_ids"][b, p]
        if T == 0:
            Zb = npd["Z"][b]
            if Zb.dtype == np.uint16:
                Zb = (Zb.astype(np.uint32) << 16).view(np.float32)
            y = np.argmax(Zb, axis=-1)  # target-argmax decoding
            assert out[:n].tolist() == y[:n].tolist()
            if n < L:
                assert g["path"][b, n - 1] != y[n - 1]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("mode", [binding.DFS_PATH_GREEDY, binding.DFS_PATH_VITERBI,
                                  binding.DFS_PATH_SAMPLE, binding.DFS_PATH_SAMPLE_JOINT])
@pytest.mark.parametrize("T", [0.0, 0.8])
def test_fused_small(lib, orc, spec, mode, T):
    data = wl.generate(spec, "cuda")
    npd = np_inputs(data)
    g = _run(data, spec, mode, T, seed=spec.seed + 100)
    o = orc.select_verify(npd["h"], npd["W"], npd["Wg"], npd["A"], npd["Bt"], npd["x0"], npd["Z"],
                          path_mode=mode, temperature=T, seed=spec.seed + 100)
    diverged = _compare(g, o, spec, list(range(spec.B)), T)
    assert diverged <= max(1, spec.B // 8)
    _invariants(g, spec, npd, T)


# Fewer LM-head CTAs, so fewer partial lists per row: the tail's merge takes groups of 1, 2 and
# 4 lists, fewer than 16 groups (every entry a candidate) and the exact merge past 64
# candidates. Up to 128 rows the list count is the CTA count, above it half.
LIST_COUNTS = [
    (SMALL[1], 4),    # 4 lists: fewer than 16 groups, 64 candidates (the buffer's size)
    (SMALL[1], 6),    # 6 lists: 96 candidates, the exact merge
    (SMALL[1], 24),   # groups of one list
    (SMALL[1], 100),  # groups of four lists
    (SMALL[2], 16),   # CTA pairs: 8 lists, the exact merge
    (SMALL[2], 60),   # 30 lists, groups of one
    (SMALL[2], 120),  # 60 lists, groups of two
]


@pytest.mark.parametrize("spec,ctas", LIST_COUNTS, ids=lambda x: getattr(x, "name", str(x)))
@pytest.mark.parametrize("mode,T", [(binding.DFS_PATH_GREEDY, 0.0), (binding.DFS_PATH_SAMPLE, 0.8)])
def test_fused_merge_list_counts(lib, orc, spec, ctas, mode, T, monkeypatch):
    monkeypatch.setenv("DFS_DEBUG_LMHEAD_CTAS", str(ctas))
    data = wl.generate(spec, "cuda")
    npd = np_inputs(data)
    g = _run(data, spec, mode, T, seed=spec.seed + 200)
    o = orc.select_verify(npd["h"], npd["W"], npd["Wg"], npd["A"], npd["Bt"], npd["x0"], npd["Z"],
                          path_mode=mode, temperature=T, seed=spec.seed + 200)
    diverged = _compare(g, o, spec, list(range(spec.B)), T)
    assert diverged <= max(1, spec.B // 8)
    _invariants(g, spec, npd, T)


def test_fused_is_deterministic(lib):
    spec = SMALL[2]
    data = wl.generate(spec, "cuda")
    a = _run(data, spec, binding.DFS_PATH_VITERBI, 0.8, 5)
    b = _run(data, spec, binding.DFS_PATH_VITERBI, 0.8, 5)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_fused_launch_count(lib):
    """One fused call launches the LM-head kernel once per group of up to 256 draft rows,
    then the tail once (target-row statistics folded into the LM-head kernel)."""
    for spec in (SMALL[1], SMALL[3]):
        data = wl.generate(spec, "cuda")
        dims = dims_for(spec)
        ws = binding.alloc_workspace(dims)
        before = binding.dfs_launch_count()
        binding.dfs_select_verify(dims, data["h"], data["W"], data["Wg"], data["A"], data["Bt"],
                                  data["x0"], data["Z"], binding.DFS_PATH_GREEDY, 0.0, 1, ws)
        torch.cuda.synchronize()
        rows = spec.B * spec.L
        assert binding.dfs_launch_count() - before == (rows + 255) // 256 + 1


def test_fused_launch_count_vocabulary_major(lib):
    """Where the drafted rows alone fit fewer 256-row groups (32 blocks of 9: 288 rows, 256
    drafted), one vocabulary-major LM-head launch replaces two."""
    spec = [s for s in SMALL if s.name == "vt_32x9"][0]
    data = wl.generate(spec, "cuda")
    dims = dims_for(spec)
    ws = binding.alloc_workspace(dims)
    before = binding.dfs_launch_count()
    binding.dfs_select_verify(dims, data["h"], data["W"], data["Wg"], data["A"], data["Bt"],
                              data["x0"], data["Z"], binding.DFS_PATH_GREEDY, 0.0, 1, ws)
    torch.cuda.synchronize()
    assert binding.dfs_launch_count() - before == 1 + 1


@pytest.mark.parametrize("name", ["fused_groups", "pairs_256rows_r512", "pairs_L16"])
@pytest.mark.parametrize("mode,T", [(binding.DFS_PATH_VITERBI, 0.0), (binding.DFS_PATH_SAMPLE, 0.8)])
def test_fused_vocabulary_major_forced(lib, orc, name, mode, T, monkeypatch):
    """The vocabulary-major LM head forced where the row-major one is the default: several
    request groups with a one-request last group, two gate tiles, 15 drafted rows a block."""
    monkeypatch.setenv("DFS_LMHEAD_VARIANT", "6")
    spec = [s for s in SMALL if s.name == name][0]
    data = wl.generate(spec, "cuda")
    npd = np_inputs(data)
    g = _run(data, spec, mode, T, seed=spec.seed + 200)
    o = orc.select_verify(npd["h"], npd["W"], npd["Wg"], npd["A"], npd["Bt"], npd["x0"], npd["Z"],
                          path_mode=mode, temperature=T, seed=spec.seed + 200)
    diverged = _compare(g, o, spec, list(range(spec.B)), T)
    assert diverged <= max(1, spec.B // 8)
    _invariants(g, spec, npd, T)


FULL = [wl.SINGLE, wl.SMALL_BATCH, wl.THROUGHPUT, wl.LONG_BLOCK]


@pytest.fixture(scope="module")
def full_size():
    """Inputs and the oracle's LM head of each full-size workload, made once per module."""
    cache = {}

    def get(orc, spec):
        if spec.name not in cache:
            cache.clear()  # one full-size workload on the device at a time
            data = wl.generate(spec, "cuda")
            npd = np_inputs(data)
            cache[spec.name] = (data, npd, oracle_head(orc, npd, spec))
        return cache[spec.name]
    return get


def _full_size_legs(spec):
    """(path mode, T, seed) of a workload: every path mode and temperature it lists, the
    sampled traversal at each T > 0 with two seeds, and the joint path draw at each T > 0."""
    code = {"greedy": binding.DFS_PATH_GREEDY, "viterbi": binding.DFS_PATH_VITERBI}
    legs = [(code[m], T, spec.seed) for m in spec.path_modes for T in spec.temperatures]
    legs += [(binding.DFS_PATH_SAMPLE, T, s) for T in spec.temperatures if T > 0
             for s in (spec.seed, spec.seed + 17)]
    legs += [(binding.DFS_PATH_SAMPLE_JOINT, T, spec.seed + 5) for T in spec.temperatures if T > 0]
    return legs


@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_fused_full_size_every_request(lib, orc, full_size, spec, monkeypatch):
    data, npd, head = full_size(orc, spec)
    names = {0: "greedy", 1: "viterbi", 2: "sampled", 3: "joint"}
    # the throughput workload also with the drafted-rows LM head forced (8 vocabulary tiles
    # per CTA pair: its threshold filter runs after the warm-up tiles)
    variants = ("0", "6") if spec is wl.THROUGHPUT else ("0",)
    for variant in variants:
        monkeypatch.setenv("DFS_LMHEAD_VARIANT", variant)
        for mode, T, seed in _full_size_legs(spec):
            g = _run(data, spec, mode, T, seed=seed)
            _invariants(g, spec, npd, T)
            o = oracle_step(orc, npd, spec, head, mode, T, seed)
            excluded = _compare(g, o, spec, range(spec.B), T,
                                name=f"{spec.name} {names[mode]} T={T} seed={seed} "
                                     f"variant={variant}")
            assert excluded <= max(1, spec.B // 4), f"{excluded} of {spec.B} excluded"
