"""Replica aggregation of the benchmark on CPU: two gloo ranks with different step times.

The decode step does not shard, so multi-GPU runs are independent replicas; the job
value is world x batch tokens over the slowest rank's step time."""
import os
import socket

import pytest
import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = bench.replica_value(10.0 + 2.0 * rank, 4, "cpu")
        out.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_replica_value_takes_slowest_rank():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == pytest.approx(12.0)
        assert value == pytest.approx(2 * 4 / 0.012)


def test_replica_value_single_process():
    import bench
    ms, value = bench.replica_value(5.0, 1, "cpu")
    assert ms == 5.0 and value == pytest.approx(200.0)
