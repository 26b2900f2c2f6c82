"""Multi-GPU runs are replicas only (rows are independent, nothing crosses
GPUs).  The host logic of that mode -- the barrier and the max-over-ranks
reduction of the step time that sets the whole-job throughput -- is checked
here with world_size 2 on the gloo backend, on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [2.0, 3.5][rank]  # per-rank mean step time
    dist.barrier()
    m = bench.replica_max(ms)
    v = bench.replica_throughput(32, world, m)
    dist.barrier()
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_replica_reduction_world_size_2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 3.5  # every rank sees the slowest replica's time
        assert v == pytest.approx(32 * 2 / 3.5e-3)


def test_replica_helpers_without_a_group():
    import bench

    assert bench.replica_max(1.25) == 1.25
    assert bench.replica_throughput(32, 1, 2.0) == pytest.approx(16000.0)
