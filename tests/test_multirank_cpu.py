"""The bench's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Replica runs are weak scaling: each rank times the same workload, the job's
time is the maximum over ranks, and the reported rate is world_size x tokens
over that time.  Only rank 0 prints; the reference arm does no work on the
other ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.cpu


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, times, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        bench.barrier()
        m = bench.max_over_ranks(times[rank], torch.device("cpu"))
        bench.barrier()
        out.put((rank, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [0.125, 0.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(out.get(timeout=10) for _ in range(2))
    assert got == {0: 0.5, 1: 0.5}


def test_max_over_ranks_without_a_process_group_is_identity():
    assert bench.max_over_ranks(3.25, "cpu") == 3.25


def test_weak_scaling_aggregate():
    # two ranks of 1e6 tokens, slowest rank 2 ms -> 1e9 tokens/s for the job
    assert bench.aggregate_rate(2, 1_000_000, 2.0) == pytest.approx(1e9)
    assert bench.aggregate_rate(1, 1_000_000, 2.0) == pytest.approx(5e8)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
