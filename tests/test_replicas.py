"""The N > 1 path of bench.py: independent replicas, no data-path collective;
the timing is the slowest rank's and the rate counts every rank's units.
Checked with two gloo ranks on the CPU (127.0.0.1)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [800.0, 1000.0][rank]  # rank 1 is the slowest
    slowest, rate = bench.replica_rate(local_ms, 500, world, True)
    dist.barrier()
    out[rank] = (slowest, rate)
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_units():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, rate = out[r]
        assert slowest == pytest.approx(1000.0)
        assert rate == pytest.approx(2 * 500 / 1000.0)


def test_single_process_rate():
    import bench

    assert bench.replica_rate(250.0, 100, 1, False) == (250.0, 0.4)
