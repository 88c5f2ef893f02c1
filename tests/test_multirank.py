"""The replica path of bench.py (N processes, one per GPU, no data-path
collective): barrier and max-over-ranks timing, exercised with world_size 2
over gloo on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    # rank r "took" 10 * (r + 1) ms for 5 steps of 8 tokens
    ms, value = bench.job_throughput(world, 8, 5, 10.0 * (rank + 1))
    out[rank] = (ms, value)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_whole_job():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # both ranks see the slowest rank's time; tokens/s covers both replicas
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == pytest.approx(20.0)
    assert value == pytest.approx(2 * 8 * 5 / 0.020)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.job_throughput(1, 8, 10, 5.0) == (5.0, 8 * 10 / 0.005)
