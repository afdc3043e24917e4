"""The multi-GPU path is replicas only (documents and heads are independent;
no collective on the data path).  What bench.py adds for N > 1 is host-side:
the slowest rank's time and the summed work.  Checked here with world size 2
over gloo on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 20.0 - rank, 3.0 * (rank + 1)]
    got = bench.reduce_max(mine, torch.device("cpu"))
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_and_job_throughput_world2():
    import bench
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True,
                           start_method="spawn")
        assert out[0] == out[1] == [11.0, 20.0, 6.0]
    # two replicas of 1e12 flops per step, 4 steps, slowest rank 2000 ms
    assert bench.job_throughput(1e12, 4, 2, 2000.0) == pytest.approx(4.0)
