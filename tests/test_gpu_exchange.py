"""The whole operator through exchange.layer on one GPU (needs a GB300).

A one-rank NCCL group: the AlltoAllv then moves this rank's rows to itself,
but goes through the same NCCL collectives, streams and host-side split
logic as on W GPUs.  The shared expert runs either beside the exchange (its
own launch) or with the routed experts (one launch); both must match the
float64 oracle within the path's tolerance and each other bit for bit.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from gpu_helpers import assert_close
from token_permute_grouped_gb300 import build, exchange
from token_permute_grouped_gb300.workloads import Workload, make_gmmX, normal_f32, rounded

pytestmark = pytest.mark.gpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.fixture(scope="module")
def nccl_group():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    yield
    dist.destroy_process_group()


@pytest.mark.parametrize("overlap", [True, False])
def test_layer_matches_oracle(orc, nccl_group, overlap):
    wl = Workload("layer_w1e4", W=1, e=4, H1=512, N1=256, dtype="bf16", routing="normal",
                  tokens_per_source=700, topk=2, bias_std=0.5, BS=300, H2=384, N2=192)
    dev = torch.device("cuda:0")
    gmmX, sc = make_gmmX(wl, seed=3, rank=0)
    gw = rounded(normal_f32(wl.e * wl.H1 * wl.N1, 4, 2) * np.float32(wl.H1 ** -0.5), (wl.e, wl.H1, wl.N1),
                 torch.bfloat16)
    mmX = rounded(normal_f32(wl.BS * wl.H2, 4, 3), (wl.BS, wl.H2), torch.bfloat16)
    mmW = rounded(normal_f32(wl.H2 * wl.N2, 4, 4) * np.float32(wl.H2 ** -0.5), (wl.H2, wl.N2), torch.bfloat16)
    gmmY, mmY, perm, ataOut, rc = exchange.layer(gmmX.to(dev), torch.from_numpy(sc).to(dev), gw.to(dev),
                                                 mmX.to(dev), mmW.to(dev), want_permute_out=True,
                                                 overlap_shared=overlap)
    torch.cuda.synchronize()
    assert torch.equal(rc.cpu(), torch.from_numpy(sc))
    assert torch.equal(ataOut.cpu().view(torch.int16), gmmX.view(torch.int16))  # one rank: rows stay in order
    ref_perm = orc.permute(1, wl.e, sc, gmmX)
    assert torch.equal(perm.cpu().view(torch.int16), ref_perm.view(torch.int16))
    _, _, groups, _ = orc.plan(1, wl.e, sc, gmmX.shape[0])
    assert_close(gmmY.cpu(), orc.grouped_matmul(groups, ref_perm, gw), "gmmY")
    assert_close(mmY.cpu(), orc.matmul(mmX, mmW), "mmY")


def test_overlap_and_single_launch_agree(nccl_group):
    wl = Workload("layer_w1e2", W=1, e=2, H1=256, N1=128, dtype="bf16", routing="normal",
                  tokens_per_source=500, topk=2, BS=256, H2=256, N2=128)
    dev = torch.device("cuda:0")
    gmmX, sc = make_gmmX(wl, seed=8, rank=0)
    gw = rounded(normal_f32(wl.e * wl.H1 * wl.N1, 9, 2) * np.float32(0.0625), (wl.e, wl.H1, wl.N1), torch.bfloat16)
    mmX = rounded(normal_f32(wl.BS * wl.H2, 9, 3), (wl.BS, wl.H2), torch.bfloat16)
    mmW = rounded(normal_f32(wl.H2 * wl.N2, 9, 4) * np.float32(0.0625), (wl.H2, wl.N2), torch.bfloat16)
    args = (gmmX.to(dev), torch.from_numpy(sc).to(dev), gw.to(dev), mmX.to(dev), mmW.to(dev))
    a = exchange.layer(*args, overlap_shared=True)
    b = exchange.layer(*args, overlap_shared=False)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
