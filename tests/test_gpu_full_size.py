"""Full-size workloads on the GPU against the oracle (needs a GB300).

Each workload runs in the launch configuration bench.py times (default path,
permuteOut not requested) and again with permuteOut.  permuteOut is compared
bit for bit in full; gmmY and mmY on sampled rows (every group's first and
last rows, the rows around each group's last tile boundary, and a seeded
random set), each checked element by element against the float64 oracle.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, assert_close, run_gpu, sample_rows
from token_permute_grouped_gb300 import build
from token_permute_grouped_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload(orc, name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, seed=0)
    gmmY, mmY, _, (st, code) = run_gpu(inp, "default", want_perm=False)
    assert st == 0, code
    # Every path and tile shape gives the same bits as the default one.
    for path, tiles in (("split", "single"), ("fused", "pair")):
        y2, m2, _, (st, code) = run_gpu(inp, path, want_perm=False, tiles=tiles)
        assert st == 0, code
        assert torch.equal(gmmY.view(torch.int16), y2.view(torch.int16)), (path, tiles)
        if mmY is not None:
            assert torch.equal(mmY.view(torch.int16), m2.view(torch.int16)), (path, tiles)
    gmmY2, mmY2, perm, (st, code) = run_gpu(inp, "default", want_perm=True)
    assert st == 0, code
    # Asking for permuteOut must not change the products.
    assert torch.equal(gmmY.view(torch.int16), gmmY2.view(torch.int16))
    if mmY is not None:
        assert torch.equal(mmY.view(torch.int16), mmY2.view(torch.int16))

    ref_perm = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut)
    assert_bits_equal(perm, ref_perm, "permuteOut")
    _, _, gr, _ = orc.plan(wl.W, wl.e, inp.recvCounts, inp.A)
    rows = sample_rows(gr, 192, seed=1)
    ref = orc.grouped_matmul(gr, ref_perm, inp.gmmWeight, rows)
    assert_close(gmmY[rows], ref, f"gmmY rows of {name}")
    if wl.BS:
        srows = sample_rows([wl.BS], 96, seed=2)
        ref = orc.matmul(inp.mmX, inp.mmWeight, srows)
        assert_close(mmY[srows], ref, f"mmY rows of {name}")
