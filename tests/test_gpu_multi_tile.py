"""The persistent GEMM with several tiles per CTA unit, every element against
the oracle (needs a GB300).

"aclnnAlltoAllvGroupedMatMul", Formula: gmmY = permuteOut x gmmWeight and
mmY = mmX x mmWeight; "Deterministic computing".  The kernels keep one CTA
(or CTA pair) per SM and walk the tile list with a fixed stride, so a unit
computes tile t, t + units, ...  These shapes have four to eight times as
many tiles as there are units.  That reaches what a one-tile-per-unit case
never does: the second TMEM accumulator, the accumulator barriers' parity
flips, the stage ring wrapping across tiles, and the epilogue of one tile
running beside the main loop of the next.  Every output element is checked
(|gpu - ref| <= 2e-2 * max(1, |ref|) against the float64 oracle), permuteOut
bit for bit, and all paths and tile shapes must give the same bits.
"""

import functools

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, assert_close, run_gpu
from token_permute_grouped_gb300 import build
from token_permute_grouped_gb300.workloads import custom_inputs, random_counts

pytestmark = pytest.mark.gpu

PATHS = ["fused", "split", "split_runs"]
TILES = ["single", "pair", "pair_k64"]

# (W, e, H1, N1, A, zero_prob, BS, H2, N2, dtype, seed)
SHAPES = {
    # About 24K routed rows in 8 x 4 runs of ~750 rows; K = 256 is two
    # 128-deep stages per tile, so the three-stage ring wraps inside and
    # across tiles.  With 256 x 256 pair tiles: ~100 m-tiles x 4 column
    # tiles plus 64 shared tiles, about six per pair unit.
    "w8e4_a24k_h256_n1024_shared4096": (8, 4, 256, 1024, 24000, 0.05, 4096, 256, 1024, "bf16", 11),
    # K = 64: one stage per tile, so tiles turn over as fast as the
    # epilogue can drain them; N = 512 gives two column tiles per row block.
    "w8e4_a60k_h64_n512_shared2048": (8, 4, 64, 512, 60000, 0.1, 2048, 64, 512, "bf16", 12),
    # fp16, empty segments, a last column tile half outside N (N1 = 1408 is
    # 5.5 tiles of 256 columns), and a shared expert with its own K and a
    # width that is not a multiple of 64.
    "w4e8_a20k_h128_n1408_fp16": (4, 8, 128, 1408, 20000, 0.25, 1000, 384, 200, "fp16", 13),
    # 32 experts of random size: nearly every group ends in a partial tile, whose
    # output blocks take the masked path while whole blocks go out by TMA
    # store; N1 = 288 gives 144-wide column tiles whose last 32-column chunk
    # runs past the tile (masked), and the shared expert's 200 columns a
    # 208-wide tile.  So full and masked blocks alternate within and across
    # a unit's tiles, which is what the epilogue's buffer reuse must survive.
    "w8e32_a40k_h128_n288": (8, 32, 128, 288, 40000, 0.1, 1500, 128, 200, "bf16", 14),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


@functools.lru_cache(maxsize=None)
def _case(name):
    W, e, H1, N1, A, zero, BS, H2, N2, dt, seed = SHAPES[name]
    rc = random_counts(W, e, A, seed, zero)
    return custom_inputs(W, e, H1, N1, rc, dt, BS, H2, N2, seed=seed)


@functools.lru_cache(maxsize=None)
def _reference(name):
    import oracle
    inp = _case(name)
    wl = inp.wl
    return oracle.Oracle().run(wl.W, wl.e, inp.recvCounts, inp.ataOut, inp.gmmWeight, inp.mmX, inp.mmWeight)


@functools.lru_cache(maxsize=None)
def _first_gpu_result(name):
    """The first path and tile shape's outputs, which every other must equal bit for bit."""
    gmmY, mmY, _, (st, code) = run_gpu(_case(name), "split", want_perm=False, tiles="single")
    assert st == 0, code
    return gmmY, mmY


def test_shapes_give_several_tiles_per_unit():
    # 152 SMs: at most 152 single-CTA units or 76 pairs.  Every shape has at
    # least four tiles per unit for each tile shape.
    for name, (W, e, H1, N1, A, zero, BS, H2, N2, dt, seed) in SHAPES.items():
        rc = np.asarray(random_counts(W, e, A, seed, zero)).reshape(W, e)
        groups = rc.sum(0)
        for tile_m, units, max_bn in ((128, 152, 256), (256, 76, 256)):
            tn1 = -(-N1 // max_bn)
            tiles = sum(-(-int(m) // tile_m) for m in groups) * tn1
            if BS:
                tiles += -(-BS // tile_m) * -(-N2 // max_bn)
            assert tiles >= 4 * units, (name, tile_m, tiles)


@pytest.mark.parametrize("want_perm", [False, True])
@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_every_element_against_oracle(name, path, tiles, want_perm):
    inp = _case(name)
    gmmY, mmY, perm, (st, code) = run_gpu(inp, path, want_perm=want_perm, guard_rows=2, sentinel=0x7FC1,
                                          tiles=tiles)
    assert st == 0, code
    ref_perm, ref_y, ref_mm = _reference(name)
    A, BS = inp.A, inp.wl.BS
    if perm is not None:
        assert_bits_equal(perm[:A], ref_perm, "permuteOut")
    assert_close(gmmY[:A], ref_y, "gmmY")
    if BS:
        assert_close(mmY[:BS], ref_mm, "mmY")
    for t, n in ((gmmY, A), (perm, A), (mmY, BS)):
        if t is not None:
            assert (t[n:].view(torch.int16) == 0x7FC1).all(), "written past the end"
    # Same fp32 accumulation order on every path and tile shape.
    y0, m0 = _first_gpu_result(name)
    assert_bits_equal(gmmY[:A], y0[:A], "gmmY vs the split/single result")
    if BS:
        assert_bits_equal(mmY[:BS], m0[:BS], "mmY vs the split/single result")
