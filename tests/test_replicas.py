"""The N > 1 path of bench.py on CPU: replicas (one process per GPU, no collective
on the data path) are timed by their slowest one, and the job's throughput counts
every replica's units. Two gloo ranks on 127.0.0.1, started with spawn."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [3.0, 5.5][rank]
        slowest = bench.max_over_ranks(local_ms, world, "cpu")
        value = bench.job_throughput(1e12, world, slowest * 1e-3)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 5.5
        assert value == pytest.approx(2 * 1e12 / 5.5e-3)


def test_one_replica_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(4.25, 1, "cpu") == 4.25
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0
