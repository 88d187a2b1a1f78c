"""The multi-GPU form of this layer is replicas only: each rank runs its own pool and batch, with no
exchange on the data path, and the bench reports all ranks' rows over the slowest rank's step.
That aggregation (one all-reduce of the step time, max over ranks) is host logic; here it runs
on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, step_ms, rows, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        value, ms = bench.replica_rate(step_ms[rank], rows, world)
        out[rank] = (value, ms)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("step_ms", [(0.100, 0.125), (0.25, 0.20)])
def test_replica_rate_is_all_rows_over_the_slowest_rank(step_ms):
    world, rows = 2, 128
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), step_ms, rows, out), nprocs=world, join=True)
    slowest = max(step_ms)
    for r in range(world):
        value, ms = out[r]
        assert ms == pytest.approx(slowest, rel=0, abs=0)  # the max, exactly (fp64 all-reduce)
        assert value == pytest.approx(world * rows / (slowest / 1e3), rel=1e-12)


def test_single_replica_needs_no_process_group():
    import bench
    value, ms = bench.replica_rate(0.1, 128, 1)
    assert ms == 0.1 and value == pytest.approx(128 / 1e-4, rel=1e-12)
