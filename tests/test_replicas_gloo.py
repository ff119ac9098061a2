"""Multi-process (world size 2, gloo, CPU) test of the bench's replica aggregation: every rank
runs the whole step on its own GPU, the job time is the slowest rank's, and the whole-job value
is (ranks x per-rank work) / that time.  No GPU is used."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [2.0, 3.5][rank]
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    value = bench.job_throughput(1e12, world, ms)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 3.5
    assert abs(value - 2 * 1e12 / 3.5e-3) < 1.0


def test_single_process_is_identity():
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.job_throughput(10.0, 1, 1000.0) == 10.0
