"""Full-size workloads on the GPU against the oracle, every element (needs a GB300).

Each workload runs in the launch configuration bench.py times (default path,
permuteOut not requested) and again with permuteOut.  permuteOut is compared
bit for bit; every row of gmmY and mmY is compared element by element with
the float64 oracle (|gpu - ref| <= 2e-2 * max(1, |ref|)), in blocks of rows
so that the float64 reference never has to be held whole.  The oracle's
products take about a minute for the largest workloads on 16 host cores.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, assert_close, run_gpu
from token_permute_grouped_gb300 import build
from token_permute_grouped_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

BLOCK_ROWS = 8192


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
    for r0 in range(0, inp.A, BLOCK_ROWS):
        rows = np.arange(r0, min(inp.A, r0 + BLOCK_ROWS), dtype=np.int64)
        ref = orc.grouped_matmul(gr, ref_perm, inp.gmmWeight, rows)
        assert_close(gmmY[r0:r0 + len(rows)], ref, f"gmmY rows {r0}.. of {name}")
    for r0 in range(0, wl.BS, BLOCK_ROWS):
        rows = np.arange(r0, min(wl.BS, r0 + BLOCK_ROWS), dtype=np.int64)
        ref = orc.matmul(inp.mmX, inp.mmWeight, rows)
        assert_close(mmY[r0:r0 + len(rows)], ref, f"mmY rows {r0}.. of {name}")
