"""Replica timing across ranks (world_size 2, gloo, CPU only).

The path shards by tokens with no exchange, so N GPUs run N independent
replicas.  The benchmark's only cross-rank logic is the barrier and the
maximum of the timed region; this checks it with two CPU processes."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    bench.barrier(w)
    elapsed = 1.0 + rank  # rank 1 is the slow one
    mx = bench.aggregate_max(elapsed, w)
    rate = bench.whole_job_rate(16384 * 10, w, mx)
    q.put((r, w, lr, mx, rate))
    dist.destroy_process_group()


def test_two_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, lr, mx, rate) in enumerate(out):
        assert (r, w, lr) == (rank, 2, rank)
        assert mx == 2.0
        assert rate == pytest.approx(16384 * 10 * 2 / 2.0)


def test_single_rank_is_identity(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.aggregate_max(3.5, 1) == 3.5
    assert bench.whole_job_rate(100, 1, 2.0) == 50.0
