"""World-size-2 gloo test of the bench's multi-rank logic on CPU: each rank
runs an independent replica, the job time is the slowest rank's and the
job's bytes are the sum over ranks (no collective on the data path)."""
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
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.5, 20.0][rank]
    nbytes = [1e9, 3e9][rank]
    t, b = bench.job_totals(ms, nbytes, world)
    dist.barrier()
    q.put((rank, t, b))
    dist.destroy_process_group()


def test_job_totals_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, b in res:
        assert t == 20.0 and b == 4e9


def test_job_totals_single_rank():
    import bench
    assert bench.job_totals(3.0, 5.0, 1) == (3.0, 5.0)
