"""bench.py's multi-process plumbing on CPU: two gloo ranks, max-over-ranks time, whole-job units."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    secs = 1.0 + rank          # rank 1 is the slow one
    value, t = bench.aggregate(secs, 100.0, w)
    q.put((rank, value, t))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_aggregate_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, value, t in res:
        assert t == 2.0                     # max over ranks
        assert value == 100.0 * world / 2.0  # units of all ranks / slowest time
