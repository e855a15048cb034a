"""Row offsets past 2^31 elements (needs a GB300 and about 15 GB of device memory).

"aclnnAlltoAllvGroupedMatMul", Shape variables: A is the sum of recvCounts,
with no small bound of its own.  Here ataOut holds 300,000 rows of 7168 bf16
values, 2.15e9 elements (4.3 GB), so every element offset past row 299,593
is beyond 2^31.  A 32-bit product of a row index and the row length anywhere
(the permute's copies, the fused path's copier warps, the epilogue's output
address) would wrap and read or write the wrong rows.

permuteOut is compared bit for bit on every row.  gmmY is compared with the
float64 oracle on sampled rows (|gpu - ref| <= 2e-2 * max(1, |ref|)): both
sides of every group boundary, the last 256 rows, and a seeded random set.
Every path runs, the default one with and without permuteOut.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, assert_close, sample_rows
from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import custom_inputs

pytestmark = pytest.mark.gpu

W, E, H1, N1 = 2, 2, 7168, 64
COUNTS = [120000, 30000, 100000, 50000]  # rank-major: (source 0, expert 0), (0, 1), (1, 0), (1, 1)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


@pytest.fixture(scope="module")
def case(orc):
    inp = custom_inputs(W, E, H1, N1, COUNTS, "bf16", seed=41)
    assert inp.A * H1 > 2**31
    ref_perm = orc.permute(W, E, inp.recvCounts, inp.ataOut)
    _, _, groups, _ = orc.plan(W, E, inp.recvCounts, inp.A)
    rows = sample_rows(groups, 600, seed=41)
    rows = np.unique(np.concatenate([rows, np.arange(inp.A - 256, inp.A)])).astype(np.int64)
    ref_y = orc.grouped_matmul(groups, ref_perm, inp.gmmWeight, rows)
    dev = torch.device("cuda:0")
    return inp, ref_perm, rows, ref_y, inp.ataOut.to(dev), inp.gmmWeight.to(dev), \
        torch.from_numpy(inp.recvCounts).to(dev)


@pytest.mark.parametrize("path,want_perm", [("default", False), ("default", True), ("split", True),
                                            ("fused", True), ("split_runs", False)])
def test_offsets_past_2_31(case, path, want_perm):
    inp, ref_perm, rows, ref_y, ata, w, rc = case
    plan = binding.Plan(W, E, inp.A, H1, N1, 0, 0, 0, torch.bfloat16, want_perm, path, device=ata.device)
    y, _, perm = plan.run(ata, rc, w)
    torch.cuda.synchronize()
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)
    if want_perm:
        assert_bits_equal(perm.cpu(), ref_perm, "permuteOut")
    del perm
    idx = torch.from_numpy(rows).to(y.device)
    assert_close(y.index_select(0, idx).cpu(), ref_y, f"gmmY sampled rows ({path})")
