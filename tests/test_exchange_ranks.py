"""The AlltoAllv front end over simulated CPU ranks (gloo; no GPU).

"aclnnAlltoAllvGroupedMatMul" page, Formula: ataOut = AlltoAllv(gmmX).  Each
of W gloo ranks draws its own gmmX and sendCounts from the sender side of the
routing model and runs token_permute_grouped_gb300.exchange.alltoallv.  On
rank r the result must be:

- recvCounts equal to what the receiver side of the same routing draw gives
  (workloads.recv_counts), with no communication involved;
- ataOut in rank-major order: every row carries a tag (source rank, global
  expert, index within its run), and the tags must read source 0's runs for
  local experts 0..e-1, then source 1's, ... with indices in order;
- after the oracle's permute and grouped product, for each local expert j,
  the product of the rows that all sources sent to global expert r*e + j
  (regenerated here from each source's seed, in source order) with
  gmmWeight[j], computed by numpy in float64.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _workload(W):
    from token_permute_grouped_gb300.workloads import Workload
    return Workload(f"exchange_w{W}e3", W=W, e=3, H1=64, N1=40, dtype="bf16", routing="normal",
                    tokens_per_source=40, topk=2, bias_std=0.7)


def _tagged_gmmX(wl, rank):
    """A source rank's gmmX with columns 0-2 set to (rank, global expert, index in run)."""
    import torch
    from token_permute_grouped_gb300.workloads import make_gmmX
    x, sc = make_gmmX(wl, seed=0, rank=rank)
    x = x.clone()
    row = 0
    for g, n in enumerate(sc):
        for i in range(int(n)):
            x[row, 0], x[row, 1], x[row, 2] = float(rank), float(g), float(i)
            row += 1
    assert row == x.shape[0]
    return x, torch.from_numpy(sc)


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from token_permute_grouped_gb300 import exchange
    from token_permute_grouped_gb300.workloads import recv_counts, rounded, normal_f32
    wl = _workload(world)
    e = wl.e
    gmmX, sc = _tagged_gmmX(wl, rank)
    ataOut, rc = exchange.alltoallv(gmmX, sc, e)
    res = {}
    res["counts"] = bool(np.array_equal(rc.numpy(), recv_counts(wl, 0, rank)))
    # Tags in rank-major order.
    want = [(w, rank * e + j, i) for w in range(world) for j in range(e) for i in range(int(rc[w * e + j]))]
    got = [tuple(int(v) for v in r[:3].tolist()) for r in ataOut.float()]
    res["order"] = got == want
    # The hot path after the exchange (oracle) against an independent product.
    gw = rounded(normal_f32(e * wl.H1 * wl.N1, 5, 2) * np.float32(wl.H1 ** -0.5), (e, wl.H1, wl.N1),
                 wl.torch_dtype)
    orc = oracle.Oracle()
    perm = orc.permute(world, e, rc.numpy(), ataOut)
    _, _, groups, _ = orc.plan(world, e, rc.numpy(), ataOut.shape[0])
    gmmY = orc.grouped_matmul(groups, perm, gw)
    sources = [_tagged_gmmX(wl, w) for w in range(world)]
    row = 0
    ok = True
    for j in range(e):
        g = rank * e + j
        blocks = []
        for x, s in sources:
            start = int(s[:g].sum())
            blocks.append(x[start:start + int(s[g])].double().numpy())
        rows = np.concatenate(blocks)
        ref = rows @ gw[j].double().numpy()
        got_j = gmmY[row:row + rows.shape[0]]
        ok &= got_j.shape == ref.shape and bool(np.allclose(got_j, ref, rtol=1e-12, atol=1e-12))
        row += rows.shape[0]
    res["product"] = ok and row == gmmY.shape[0]
    res["A"] = int(ataOut.shape[0])
    out[rank] = res
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_alltoallv_gives_rank_major_ataOut(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(out)
    total = 0
    for r in range(world):
        assert res[r]["counts"], r
        assert res[r]["order"], r
        assert res[r]["product"], r
        total += res[r]["A"]
    wl = _workload(world)
    assert total == world * wl.tokens_per_source * wl.topk  # every selection lands on exactly one rank


def test_sender_and_receiver_counts_agree():
    from token_permute_grouped_gb300.workloads import W8E4, WORKLOADS, recv_counts, send_counts
    for name in (W8E4, "dsv3_w32e8_h7168_n4096_shared4096"):
        wl = WORKLOADS[name]
        sends = [send_counts(wl, 0, w) for w in range(wl.W)]
        for r in (0, wl.W - 1):
            rc = recv_counts(wl, 0, r)
            want = np.concatenate([sends[w][r * wl.e:(r + 1) * wl.e] for w in range(wl.W)])
            assert np.array_equal(rc, want)
        assert all(int(s.sum()) == wl.tokens_per_source * wl.topk for s in sends)
