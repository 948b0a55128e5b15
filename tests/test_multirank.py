"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

With N GPUs every rank runs its own batch (weak scaling, no data-path
collective); the only cross-rank operations are the barrier around the timed
region and the max over ranks of the elapsed time.  This test runs those two
with two gloo ranks on 127.0.0.1.
"""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(ws)
        slowest = bench.max_over_ranks(1.5 + rank, ws)  # rank 1 is the slow one
        results[rank] = slowest
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_rank_barrier_and_max_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        assert dict(results) == {0: 2.5, 1: 2.5}
