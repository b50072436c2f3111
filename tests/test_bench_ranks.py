"""Multi-rank aggregation of bench.py (replicas only: max time over ranks, sum
of work over ranks), exercised with world_size 2 on the gloo backend."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.combine_ranks(10.0 + 5.0 * rank, 4 * (rank + 1))
    out[rank] = (ms, units)
    dist.destroy_process_group()


def test_combine_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert out[0] == out[1] == (15.0, 12)


def test_combine_ranks_single_process():
    import bench
    assert bench.combine_ranks(3.5, 7) == (3.5, 7)
