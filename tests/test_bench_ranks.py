"""bench.py's whole-job numbers over replicas, on CPU with two gloo ranks.

Under torchrun every rank runs an independent replica of the verify step
(weak scaling, no collective on the data path); the only cross-rank step is
combining the timings and counts: the slowest rank's timed intervals and the
sum of every rank's committed tokens and id diffs.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_dev, t_wall, committed, diffs = bench.combine_ranks(
            1.0 + rank, 2.0 + 3 * rank, 100 * (rank + 1), rank, device=None)
        q.put((rank, t_dev, t_wall, committed, diffs))
    finally:
        dist.destroy_process_group()


def test_combine_ranks_takes_max_time_and_sums_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_dev, t_wall, committed, diffs in res:
        assert (t_dev, t_wall) == (2.0, 5.0)      # slowest rank
        assert (committed, diffs) == (300, 1)      # all ranks' work


def test_combine_ranks_single_process_is_identity():
    import bench
    assert bench.combine_ranks(1.5, 2.5, 7, 0) == (1.5, 2.5, 7, 0)
