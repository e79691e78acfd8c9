"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the
timing reduction takes the slowest rank and the whole-job throughput counts
every rank's work.  No GPU is involved."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_setup() == (world, rank, rank)
        mine = [10.0 + rank, 20.0 - rank]  # rank 1 is slower on the first figure
        got = bench.reduce_max_over_ranks(mine)
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == [11.0, 20.0]

    import bench

    # 2 ranks x 3 steps x 1e12 FLOP in 1.5 s (the slowest rank) = 4 TFLOPS
    assert bench.job_tflops(2, 1e12, 3, 1500.0) == pytest.approx(4.0)


def test_single_process_reduction_is_identity():
    import bench

    assert bench.reduce_max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
