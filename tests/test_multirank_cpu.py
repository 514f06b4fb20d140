"""Host logic of the multi-GPU bench path, as world_size-2 gloo ranks on the CPU: each rank
verifies its own batch (no data-path exchange), timing is the max over ranks, the reported
value aggregates the rows of all ranks."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = bench.shard_workload(1, rank)
    elapsed = 10.0 + 5.0 * rank                       # rank 1 is the slow one
    mx = bench.all_reduce_max(elapsed, world, "cpu")
    digest = float(wl.target.astype(np.float64).sum())
    got = [None] * world
    dist.all_gather_object(got, (wl.B, wl.gmax, wl.V, digest))
    q.put((rank, mx, got, bench.aggregate_rate(world, wl.verified_rows(), 100, mx)))
    dist.destroy_process_group()


def test_two_rank_sharding_and_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, got, value in res:
        assert mx == 15.0                              # max over ranks
        (b0, g0, v0, d0), (b1, g1, v1, d1) = got
        assert (b0, g0, v0) == (b1, g1, v1) == (8, 4, 1024)
        assert d0 != d1                                # each rank has its own batch
        assert abs(value - 2 * 32 * 100 / 0.015) < 1e-6

