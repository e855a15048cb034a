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


@pytest.fixture(scope="module")
def mx_case(orc):
    from token_permute_grouped_gb300.workloads import Workload, make_mx_inputs
    wl = Workload("mx_offsets", W=W, e=E, H1=H1, N1=N1, dtype="bf16", routing="given")
    inp = make_mx_inputs(wl, seed=42, qtype="e4m3fn", recvCounts=np.asarray(COUNTS, np.int32))
    assert inp.A * H1 > 2**31
    perm_q = orc.permute(W, E, inp.recvCounts, inp.ataOut_q.view(torch.int16)).view(torch.uint8)
    perm_s = orc.permute(W, E, inp.recvCounts, inp.ataOut_s.view(torch.int16)).view(torch.uint8)
    _, _, groups, _ = orc.plan(W, E, inp.recvCounts, inp.A)
    rows = sample_rows(groups, 400, seed=42)
    rows = np.unique(np.concatenate([rows, np.arange(inp.A - 256, inp.A)])).astype(np.int64)
    ref_y = orc.mx_grouped_matmul(groups, perm_q, perm_s, inp.gmmWeight_q, inp.gmmWeight_s, 0, 0, rows)
    return inp, perm_q, perm_s, rows, ref_y


@pytest.mark.parametrize("tiles,want_perm", [("pair", False), ("pair", True), ("single", False)])
def test_mx_offsets_past_2_31(mx_case, tiles, want_perm):
    inp, perm_q, perm_s, rows, ref_y = mx_case
    dev = torch.device("cuda:0")
    plan = binding.MxPlan(W, E, inp.A, H1, N1, 0, 0, 0, "e4m3fn", want_perm, dev, tiles)
    y, _, pq, ps = plan.run(inp.ataOut_q.to(dev), inp.ataOut_s.to(dev), torch.from_numpy(inp.recvCounts).to(dev),
                            inp.gmmWeight_q.to(dev), inp.gmmWeight_s.to(dev))
    torch.cuda.synchronize()
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)
    if want_perm:
        assert torch.equal(pq.cpu(), perm_q) and torch.equal(ps.cpu(), perm_s)
    idx = torch.from_numpy(rows).to(dev)
    assert_close(y.index_select(0, idx).cpu(), ref_y, f"mx gmmY sampled rows ({tiles})")
