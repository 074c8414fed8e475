"""The N > 1 bench path on CPU: two gloo ranks (no GPU).

The hot path has no exchange step (each GPU re-quantizes its own replica of the
weights and runs its own rollouts), so bench.py runs independent replicas; its
only cross-rank logic is the barrier around the timed region and the MAX over
ranks of every timing, checked here with world_size 2.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(world)
        got = bench.max_over_ranks(1.5 + 2.0 * rank, world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=10) for _ in range(2))
    assert results == {0: 3.5, 1: 3.5}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.25, 1) == 2.25
    bench.barrier(1)


def test_bench_starts_its_own_replicas(tmp_path):
    """`bench.py --gpus 2` with no launcher starts two local ranks itself (torchrun);
    exactly one line comes out (rank 0), and it reports both ranks.  The reference arm
    is used: it needs no GPU (rank 0 times the oracle, rank 1 exits without work)."""
    import json
    import subprocess
    import sys

    import bench
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    p = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3", "--config", "sana", "--rows", "256"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=str(tmp_path))
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2
