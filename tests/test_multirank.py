"""Host logic of the N>1 benchmark path with world_size-2 gloo ranks on CPU.

Each rank runs an independent replica of the workload (requests are
independent; no collective on the data path); the job reports the slowest
rank's time and the units of all ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        ms, kvb, rows = bench.aggregate_ranks(10.0 + 5 * r, 1000.0 * (r + 1), 7.0 * (r + 1), w, "cpu")
        wl = bench.make_workload(1, r, reqs=3)
        q.put((r, ms, kvb, rows, wl.steps[0].seq_lens.tolist(), wl.pool_shape()))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_and_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=120) for _ in range(2)])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, ms, kvb, rows, lens, shape in res:
        assert ms == 15.0            # the slowest rank
        assert kvb == 3000.0         # units of both ranks
        assert rows == 21.0
    # each rank is its own replica: same shapes, different seeded data
    assert res[0][5][1:] == res[1][5][1:]
    assert res[0][4] != res[1][4]


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate_ranks(3.5, 10, 2, 1, "cpu") == (3.5, 10.0, 2.0)
