"""The multi-GPU path of bench.py is replicas only: each rank runs the whole
layer on its own tokens and the job time is the slowest rank's.  These CPU
tests run the same reductions with world size 2 over gloo."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 10.0][rank]
    flops = [3e12, 3e12][rank]
    tmax = bench.reduce_max(ms, world)
    fsum = bench.reduce_sum(flops, world)
    bench.barrier(world)
    q.put((rank, tmax, fsum))
    dist.destroy_process_group()


def test_replica_reductions_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tmax, fsum in res:
        assert tmax == 12.5  # the slowest rank sets the job time
        assert fsum == 6e12  # work of all ranks
    # whole-job value as bench.py computes it
    assert fsum / (tmax / 1e3) / 1e12 == pytest.approx(480.0)
