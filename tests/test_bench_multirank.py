"""bench.py's multi-rank timing logic on CPU: two gloo ranks (no GPU).

Checks the barrier + max-over-ranks timing and the sum of work over ranks
that the N-GPU line is built from, with a rank that is deliberately slower.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import time

    import torch
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    dev = torch.device("cpu")
    delay = 0.05 * (rank + 1)  # rank 1 is twice as slow
    dt, dt_max = bench.timed_region(lambda i: time.sleep(delay), 4, world, dev, lambda: None)
    work = bench.reduce_sum(10.0 * (rank + 1), world, dev)
    out[rank] = (dt, dt_max, work)
    torch.distributed.destroy_process_group()


def test_two_rank_max_over_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    dt0, max0, work0 = res[0]
    dt1, max1, work1 = res[1]
    assert max0 == pytest.approx(max1)
    assert max0 >= 4 * 0.1 * 0.95      # the slow rank's four steps
    assert max0 == pytest.approx(max(dt0, dt1))
    assert work0 == work1 == 30.0
