"""bench.py's multi-rank aggregation on CPU ranks (gloo, world size 2).

Under torchrun every rank runs an independent replica; the reported value is
all ranks' tokens over the slowest rank's time.  This runs the same reduction
the bench uses with two CPU processes."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]          # rank 1 is the slow one
        units = [800, 800][rank]
        out[rank] = bench.aggregate(dist, ms, units)
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, units = res[r]
        assert ms == 20.0 and units == 1600     # max time, summed tokens, on every rank
    assert 1600 / (20.0 / 1e3) == 80000.0


def test_aggregate_single_rank_passthrough():
    import bench
    assert bench.aggregate(None, 3.0, 7) == (3.0, 7)
