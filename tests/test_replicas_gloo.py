"""Multi-process host logic of the benchmark's replica mode, on CPU with the
gloo backend (world size 2): each rank times its own replica, the job takes
the slowest rank's step time and counts every rank's tokens."""
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
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.replica_result(10.0 + 5.0 * rank, 32)
    assert bench._dist() == (world, rank, 0)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_timing_takes_max_over_ranks_and_sums_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 15.0                       # slowest rank
        assert value == pytest.approx(32 * world / 15e-3)


def test_single_process_is_unchanged():
    import bench
    assert bench.replica_result(8.0, 32) == (8.0, 32 / 8e-3)
