"""Multi-rank aggregation of bench.py on CPU: two gloo ranks (world size 2).

The fold shards by rows with no data-path collective; bench.py only uses the
process group to barrier around the timed region and to take the max (time)
and sum (e2e throughput) over ranks. This checks that path without a GPU.
"""
from __future__ import annotations

import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    ctx = bench.DistCtx()
    ms = [3.0, 5.0][rank]                     # rank 1 is the slower one
    ctx.barrier()
    ms_max = ctx.max(ms)
    total = ctx.sum(100.0 * (rank + 1))
    value, ms_per_step = bench.aggregate(64, ms_max, 10, ctx.world)
    out[rank] = (ms_max, total, value, ms_per_step, ctx.backend)
    ctx.close()


def test_two_gloo_ranks_aggregate_weak_scaling():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        ms_max, total, value, ms_per_step, backend = res[r]
        assert backend == "gloo"
        assert ms_max == 5.0 and total == 300.0
        # all ranks' rows (2 x 64 x 10) over the slowest rank's time
        assert abs(value - 2 * 64 * 10 / 5e-3) < 1e-6 * value
        assert ms_per_step == 0.5
