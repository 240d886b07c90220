"""The bench's multi-rank aggregation (one group per rank, replicas only):
max over ranks of the timed region, divided by the groups all ranks did.
Runs as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    t_local = 2.0 if rank == 0 else 3.5
    t, v = bench.aggregate(t_local, steps=5, world=world, pg=dist)
    q.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in out:
        assert t == 3.5
        assert v == pytest.approx(3.5 / (5 * 2))


def test_aggregate_single_rank():
    import bench

    assert bench.aggregate(1.5, 3, 1) == (1.5, 0.5)
