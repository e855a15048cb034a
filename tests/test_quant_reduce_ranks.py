"""Quantised reduce-scatter over simulated CPU ranks (gloo; no GPU).

"aclnnQuantReduceScatter" page, Formula: each rank's codes x and scales go
through an AllToAll, and the Reduce sums the ranks' dequantised pieces.  Each
of W gloo ranks holds x [BS, H] and its scales, splits them into W row blocks
and exchanges them with all_to_all_single: rank r receives block r of every
rank, which is exactly the [W, BS/W, H] input the reduce takes (source rank w
at index w).  The oracle's reduce over that input must equal, element by
element, block r of an independent reduce-scatter: every rank dequantises
its whole x in float64 and an all_reduce sums them.  With E8M0 scales (powers
of two from 2^-10 to 2^6) every term and sum is exact in float64, so the two
must be equal; with float32 scales the terms carry 28 significant bits and the
two sums add them in different orders, so they agree to W float64 roundings
of sum_w |term|.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
QCODE = {"e4m3fn": 0, "e5m2": 1, "int8": 2}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, BS, H, qtype, mode, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from token_permute_grouped_gb300.workloads import quant_reduce_inputs
    orc = oracle.Oracle()
    # This rank's x [BS, H] and scales, seeded by rank (a 1-rank draw of BS rows).
    x, sc = quant_reduce_inputs(1, BS, H, qtype, mode, seed=100 + rank)
    x, sc = x[0], sc[0]
    recv_x = torch.empty_like(x)
    recv_sc = torch.empty_like(sc)
    dist.all_to_all_single(recv_x, x)        # row block r of every rank, in rank order
    dist.all_to_all_single(recv_sc, sc)
    rows = BS // world
    mine = orc.quant_reduce(recv_x.reshape(world, rows, H).numpy(), recv_sc.reshape(world, rows, -1).numpy(),
                            QCODE[qtype], 0 if mode == "mx" else 1)
    # Independent: dequantise all of x here, sum over ranks, keep block r.
    group = 32 if mode == "mx" else 128
    v = orc.decode8(QCODE[qtype], x.numpy())
    s = orc.decode8(3, sc.numpy()) if mode == "mx" else sc.numpy().astype(np.float64)
    deq = torch.from_numpy(v * np.repeat(s, group, axis=1))
    mag = deq.abs()
    dist.all_reduce(deq)
    dist.all_reduce(mag)
    want = deq[rank * rows:(rank + 1) * rows].numpy()
    S = mag[rank * rows:(rank + 1) * rows].numpy()
    ok = np.array_equal(mine, want) if mode == "mx" else bool((np.abs(mine - want) <= world * 2.0 ** -52 * S).all())
    out[rank] = (bool(ok), float(np.abs(mine - want).max()), mine.shape)
    dist.destroy_process_group()


@pytest.mark.parametrize("world,qtype,mode", [(2, "e4m3fn", "mx"), (4, "e5m2", "mx"), (2, "int8", "group128"),
                                              (4, "e4m3fn", "group128")])
def test_alltoall_then_reduce_is_reduce_scatter(world, qtype, mode):
    BS, H = 8 * world, 1024
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, BS, H, qtype, mode, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        equal, maxdiff, shape = res[r]
        assert shape == (BS // world, H)
        assert equal, (r, maxdiff)
