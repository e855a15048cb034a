"""Block-scaled FP8 (mx) grouped GEMM on the GPU against the float64 oracle (needs a GB300).

include/a2av_gmm_mx.h: gmmY = permuteOut x gmmWeight and mmY = mmX x mmWeight
with E4M3FN/E5M2 codes and one E8M0 scale per 32 elements along K
("aclnnQuantReduceScatter" page, Constraints, for the format).  permuteOut
(codes and scales) must be bit-exact; gmmY and mmY must satisfy the path's
tolerance |gpu - ref| <= 2e-2 * max(1, |ref|) against the oracle's float64
sum.  Where every partial sum is a small integer the fp32 accumulator is
exact in any order, so the output must be the bf16 rounding of the oracle's
value, bit for bit; the scale-layout cases are built that way.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close
from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import (W8E4, WORKLOADS, make_mx_inputs, mx_quantize,
                                                   random_counts, MxInputs, Workload)

pytestmark = pytest.mark.gpu
QCODE = {"e4m3fn": 0, "e5m2": 1}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


TILES = ["single", "pair"]


def run_mx(inp: MxInputs, want_perm=False, tiles="default"):
    dev = torch.device("cuda:0")
    wl = inp.wl
    plan = binding.MxPlan(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, inp.qtype, want_perm, dev, tiles)
    d = lambda t: None if t is None else t.to(dev)
    out = plan.run(d(inp.ataOut_q), d(inp.ataOut_s), torch.from_numpy(inp.recvCounts).to(dev),
                   d(inp.gmmWeight_q), d(inp.gmmWeight_s), d(inp.mmX_q), d(inp.mmX_s), d(inp.mmWeight_q),
                   d(inp.mmWeight_s))
    torch.cuda.synchronize()
    st = binding.a2av_gmm_read_device_status(plan.workspace)
    return [None if t is None else t.cpu() for t in out], st


def reference(orc, inp: MxInputs, rows=None, shared_rows=None):
    """(expert-major codes, scales, gmmY rows, mmY rows) from the oracle."""
    wl = inp.wl
    q = QCODE[inp.qtype]
    perm_q = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut_q.view(torch.int16)).view(torch.uint8)
    perm_s = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut_s.view(torch.int16)).view(torch.uint8)
    _, _, groups, _ = orc.plan(wl.W, wl.e, inp.recvCounts, inp.A)
    y = orc.mx_grouped_matmul(groups, perm_q, perm_s, inp.gmmWeight_q, inp.gmmWeight_s, q, q, rows) if inp.A else None
    m = None
    if wl.BS:
        m = orc.mx_grouped_matmul([wl.BS], inp.mmX_q, inp.mmX_s, inp.mmWeight_q[None], inp.mmWeight_s[None], q, q,
                                  shared_rows)
    return perm_q, perm_s, y, m


def _custom(W, e, H1, N1, rc, qtype="e4m3fn", BS=0, H2=0, N2=0, seed=0):
    wl = Workload(f"mx_w{W}e{e}", W=W, e=e, H1=H1, N1=N1, dtype="bf16", routing="uniform",
                  BS=BS, H2=H2, N2=N2)
    return make_mx_inputs(wl, seed=seed, qtype=qtype, recvCounts=np.asarray(rc, np.int32))


def _ones_case(sa, sw, A=256, H1=512, N1=256):
    """Every code E4M3 1.0 with the given scale codes: out[m][n] = 32 sum_b 2^(sa[m,b]+sw[n,b]-254)."""
    wl = Workload("mx_ones", W=1, e=1, H1=H1, N1=N1, dtype="bf16", routing="uniform")
    return MxInputs(wl, "e4m3fn", np.array([A], np.int32), torch.full((A, H1), 0x38, dtype=torch.uint8),
                    sa, torch.full((1, N1, H1), 0x38, dtype=torch.uint8), sw)


def _layout_cases():
    A, N1, kb = 256, 256, 16
    one_a = torch.full((A, kb), 127, dtype=torch.uint8)
    one_w = torch.full((1, N1, kb), 127, dtype=torch.uint8)
    rows = (127 + torch.arange(A) % 5)[:, None].repeat(1, kb).to(torch.uint8)
    cols = (127 + torch.arange(N1) % 5)[None, :, None].repeat(1, 1, kb).to(torch.uint8)
    blocks_a = (127 + torch.arange(kb) % 4)[None, :].repeat(A, 1).to(torch.uint8)
    blocks_w = (127 + torch.arange(kb) % 4)[None, None, :].repeat(1, N1, 1).to(torch.uint8)
    mixed = (120 + (torch.arange(A)[:, None] + 3 * torch.arange(kb)[None, :]) % 11).to(torch.uint8)
    return {"unit": (one_a, one_w), "per_row": (rows, one_w), "per_column": (one_a, cols),
            "per_block_a": (blocks_a, one_w), "per_block_b": (one_a, blocks_w), "row_and_block": (mixed, blocks_w)}


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("case", list(_layout_cases()))
def test_scale_placement_exact(orc, case, tiles):
    # Which E8M0 byte scales which row, column and K-block: every output is
    # an exact small power-of-two sum, so the bf16 result must be bit-exact.
    sa, sw = _layout_cases()[case]
    inp = _ones_case(sa, sw, H1=512)
    (y, _, _, _), st = run_mx(inp, tiles=tiles)
    assert st[0] == 0, st
    _, _, ref, _ = reference(orc, inp)
    want = torch.from_numpy(ref).to(torch.bfloat16)
    assert torch.equal(y.view(torch.int16), want.view(torch.int16)), (y[:2, :4], want[:2, :4])


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("qtype", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("W,e,H1,N1,A,zero,BS,H2,N2", [
    (2, 2, 512, 128, 300, 0.0, 0, 0, 0),
    (4, 3, 1024, 200, 700, 0.3, 100, 512, 136),
    (8, 4, 2048, 256, 1500, 0.1, 257, 1024, 384),
    # The largest H1 below 65536 that is a multiple of 512: 254 stages of 256 codes.
    (2, 2, 65024, 64, 200, 0.0, 0, 0, 0),
])
def test_matches_oracle(orc, qtype, W, e, H1, N1, A, zero, BS, H2, N2, tiles):
    rc = random_counts(W, e, A, seed=A + W, zero_prob=zero)
    inp = _custom(W, e, H1, N1, rc, qtype, BS, H2, N2, seed=W)
    (y, m, _, _), st = run_mx(inp, tiles=tiles)
    assert st[0] == 0, st
    _, _, ref_y, ref_m = reference(orc, inp)
    assert_close(y, ref_y, "gmmY")
    if BS:
        assert_close(m, ref_m, "mmY")


@pytest.mark.parametrize("tiles", TILES)
def test_shared_expert_only(orc, tiles):
    # No routed rows (A = 0): the prep kernel writes only the shared expert's
    # scale atoms and the GEMM runs only the shared tiles.
    inp = _custom(4, 2, 512, 128, [0] * 8, "e4m3fn", BS=300, H2=1024, N2=200, seed=9)
    (y, m, _, _), st = run_mx(inp, tiles=tiles)
    assert st[0] == 0, st
    _, _, _, ref_m = reference(orc, inp)
    assert_close(m, ref_m, "mmY")


def test_permute_out_bit_exact_and_same_products(orc):
    rc = random_counts(4, 2, 600, seed=5, zero_prob=0.25)
    inp = _custom(4, 2, 1024, 128, rc, "e4m3fn", seed=5)
    (y, _, pq, ps), st = run_mx(inp, want_perm=True)
    assert st[0] == 0, st
    ref_q, ref_s, _, _ = reference(orc, inp)
    assert torch.equal(pq, ref_q) and torch.equal(ps, ref_s)
    (y2, _, _, _), st = run_mx(inp, want_perm=False)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    # The other tile shape gives the same bits (fp32 sums of the same K
    # blocks in the same order).
    (y3, _, _, _), st = run_mx(inp, tiles="single")
    assert st[0] == 0 and torch.equal(y3.view(torch.int16), y.view(torch.int16))


def test_integer_products_bit_exact(orc):
    # Codes of small integers (E4M3 1, 2, 3, 4 and negatives) at unit scale:
    # every partial sum is an integer below 2^24, exact in fp32 in any order.
    rng = np.random.default_rng(4)
    vals = np.array([0x38, 0x40, 0x44, 0x48, 0xB8, 0xC0, 0x00], np.uint8)
    rc = np.array([40, 0, 90, 30], np.int32)  # W = 2, e = 2
    wl = Workload("mx_int", W=2, e=2, H1=512, N1=64, dtype="bf16", routing="uniform")
    A = int(rc.sum())
    inp = MxInputs(wl, "e4m3fn", rc, torch.from_numpy(vals[rng.integers(0, 7, (A, 512))]),
                   torch.full((A, 16), 127, dtype=torch.uint8),
                   torch.from_numpy(vals[rng.integers(0, 7, (2, 64, 512))]), torch.full((2, 64, 16), 127, dtype=torch.uint8))
    for tiles in TILES:
        (y, _, _, _), st = run_mx(inp, tiles=tiles)
        assert st[0] == 0, st
        _, _, ref, _ = reference(orc, inp)
        assert torch.equal(y.view(torch.int16), torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16)), tiles


def test_bad_counts_are_reported(orc):
    inp = _custom(2, 2, 512, 128, [10, 20, 30, 40], seed=1)
    inp.recvCounts = np.array([10, 20, 30, 41], np.int32)  # sums to A + 1
    _, st = run_mx(inp)
    assert st[0] == 6 and st[1] & 1, st  # A2AV_ERR_DEVICE_CHECK, bad-counts bit in the status word


def test_full_size_headline(orc):
    # The 8-rank x 4-expert workload in mx form, compared on sampled rows.
    inp = make_mx_inputs(WORKLOADS[W8E4], seed=0, qtype="e4m3fn")
    (y, m, _, _), st = run_mx(inp)
    assert st[0] == 0, st
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, inp.A - 1], rng.integers(0, inp.A, 48)]))
    srows = np.unique(np.concatenate([[0, inp.wl.BS - 1], rng.integers(0, inp.wl.BS, 16)]))
    _, _, ref_y, ref_m = reference(orc, inp, rows=rows, shared_rows=srows)
    assert_close(y[rows], ref_y, "gmmY")
    assert_close(m[srows], ref_m, "mmY")


_MULTI = {}

# (W, e, H1, N1, A, zero_prob, BS, H2, N2, seed)
MULTI_CASES = {
    # About 24K routed rows and a 4096-row shared expert: with 256 x 256 pair
    # tiles about six tiles per pair unit, with 128 x 128 single tiles about
    # eleven per CTA.  Each unit therefore reuses its accumulator and scale
    # columns across tiles and wraps its stage ring many times.
    "w8e4_a24k_n1024": (8, 4, 512, 1024, 24000, 0.05, 4096, 512, 1024, 21),
    # 32 experts of random size, N1 = 288 and N2 = 200: partial row tiles and
    # a last column tile only partly inside N, so blocks that go out by TMA
    # store and blocks that take the masked path alternate in every unit.
    "w8e32_a40k_n288": (8, 32, 512, 288, 40000, 0.1, 1500, 512, 200, 22),
}


def _multi_tile_case(name):
    if name not in _MULTI:
        W, e, H1, N1, A, zero, BS, H2, N2, seed = MULTI_CASES[name]
        rc = random_counts(W, e, A, seed=seed, zero_prob=zero)
        _MULTI[name] = {"inp": _custom(W, e, H1, N1, rc, "e4m3fn", BS=BS, H2=H2, N2=N2, seed=seed)}
    return _MULTI[name]


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("name", sorted(MULTI_CASES))
def test_multi_tile_every_element(orc, name, tiles):
    case = _multi_tile_case(name)
    inp = case["inp"]
    (y, m, _, _), st = run_mx(inp, tiles=tiles)
    assert st[0] == 0, st
    if "ref" not in case:
        case["ref"] = reference(orc, inp)
        case["first"] = (y, m)
    _, _, ref_y, ref_m = case["ref"]
    assert_close(y, ref_y, "gmmY")
    assert_close(m, ref_m, "mmY")
    # Both tile shapes give the same bits.
    y0, m0 = case["first"]
    assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    assert torch.equal(m.view(torch.int16), m0.view(torch.int16))
