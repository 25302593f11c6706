"""The replica (N > 1) timing path of bench.py on CPU with gloo, world_size 2: every rank runs its
own chain, the job time is the slowest rank's, and the work of all ranks is summed."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = bench.aggregate(local_ms=10.0 * (rank + 1), bytes_per_step=1_000_000, steps=50, world=world)
    bench.barrier(world)
    out[rank] = res
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        assert res[r]["ms"] == pytest.approx(20.0)
        assert res[r]["ms_per_step"] == pytest.approx(20.0 / 50)
        assert res[r]["gbs"] == pytest.approx(2 * 50 * 1_000_000 / 0.020 / 1e9)
