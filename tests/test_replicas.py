"""Host-side logic of the multi-GPU replica benchmark, run as two gloo ranks
on the CPU: the job time is the slowest rank's, the value counts every
rank's work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = [1.5, 2.5][rank]              # rank 1 is the slow one
        worst = bench.max_over_ranks(seconds)
        value = bench.job_value(units_per_rank=10.0, world=world, max_seconds=worst)
        bench.barrier()
        with open(os.path.join(outdir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{worst} {value}")
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for rank in range(world):
        worst, value = map(float, open(tmp_path / f"rank{rank}.txt").read().split())
        assert worst == pytest.approx(2.5)
        assert value == pytest.approx(10.0 * 2 / 2.5)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_value(4.0, 1, 2.0) == 2.0
