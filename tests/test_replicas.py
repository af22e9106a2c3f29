"""Replica plumbing of the benchmark on two CPU ranks (gloo): the step partitions by
request, so ranks exchange nothing on the data path; torch.distributed carries only the
start barrier and the reductions of the measured times and unit counts."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from draft_speculative_decoding_gb300 import replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, local = replicas.init(backend="gloo")
    replicas.barrier()
    # rank k processed k+1 units of work in 0.5*(k+1) seconds
    res = {
        "info": (r, w, local),
        "max": replicas.max_over_ranks(10.0 + r),
        "sum": replicas.sum_over_ranks(1.0 + r),
        "rate": replicas.job_throughput(1.0 + r, 0.5 * (1 + r)),
        "shard": list(replicas.shard(11, w, r)),
    }
    replicas.barrier()
    replicas.finalize()
    out.put((rank, res))


def test_two_rank_reductions_and_shards():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(k, world, port, q)) for k in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for k in range(world):
        assert got[k]["info"] == (k, world, k)
        assert got[k]["max"] == 11.0  # the slowest rank sets the time
        assert got[k]["sum"] == 3.0
        assert got[k]["rate"] == pytest.approx(3.0 / 1.0)  # all units over the slowest time
    assert got[0]["shard"] + got[1]["shard"] == list(range(11))  # disjoint, covering, in order


@pytest.mark.parametrize("n,world", [(0, 3), (5, 1), (7, 3), (32, 8), (3, 8)])
def test_shard_partitions(n, world):
    parts = [list(replicas.shard(n, world, k)) for k in range(world)]
    assert sum(parts, []) == list(range(n))
    sizes = [len(p) for p in parts]
    assert max(sizes) - min(sizes) <= 1


def test_single_process_is_identity():
    assert replicas.max_over_ranks(2.5) == 2.5
    assert replicas.job_throughput(32, 0.5) == 64.0


def test_reference_arm_prints_once_under_torchrun(tmp_path):
    """bench.py --impl reference under a two-rank launch: rank 0 alone runs the oracle and
    prints one JSON line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "tiny_B1_L4_V1024_d256_r32_fp32"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
