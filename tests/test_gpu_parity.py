"""CUDA path against the CPU oracle, through the C ABI (needs a GB300).

permuteOut must match bit for bit; gmmY and mmY must satisfy
|gpu - ref| <= 2e-2 * max(1, |ref|) against the float64 oracle, element by
element.  Inputs are the seeded synthetic workloads and explicit edge cases.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, assert_close, check_full, rne_to, run_gpu
from token_permute_grouped_gb300 import build
from token_permute_grouped_gb300.workloads import WORKLOADS, SMALL, Inputs, custom_inputs, make_inputs

pytestmark = pytest.mark.gpu

PATHS = ["fused", "split", "split_runs"]
TILES = ["single", "pair", "pair_k64"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


@pytest.mark.parametrize("path", PATHS + ["default"])
@pytest.mark.parametrize("want_perm", [True, False])
def test_tiny_workload(orc, path, want_perm):
    inp = make_inputs(WORKLOADS[SMALL])
    gmmY, mmY, perm, (st, code) = run_gpu(inp, path, want_perm)
    assert st == 0, code
    check_full(orc, inp, gmmY, mmY, perm)


# (W, e, H1, N1, counts, BS, H2, N2, dtype): several tiles, ragged tails,
# empty segments and groups, tile widths that are not multiples of 64.
EDGE = {
    "single_expert_plain_matmul": (1, 1, 256, 256, [300], 0, 0, 0, "bf16"),
    "ragged_multi_tile": (4, 8, 512, 384, None, 300, 320, 200, "bf16"),
    "empty_groups_and_segments": (3, 5, 128, 96, [0, 5, 0, 129, 0, 0, 0, 0, 1, 0, 0, 7, 0, 128, 0], 0, 0, 0, "bf16"),
    "one_row_groups": (2, 4, 64, 64, [1, 0, 1, 0, 0, 1, 0, 1], 1, 64, 64, "fp16"),
    "k_tail_not_multiple_of_64": (2, 3, 200, 136, None, 130, 72, 40, "bf16"),
    "narrow_n": (2, 2, 128, 8, [3, 130, 60, 1], 5, 64, 24, "bf16"),
    "bn_240_like_1408": (2, 2, 128, 1408, [100, 150, 29, 2], 0, 0, 0, "bf16"),
    "no_routed_rows_shared_only": (4, 2, 128, 128, [0] * 8, 257, 256, 136, "bf16"),
    "fp16_mixed": (8, 4, 256, 512, None, 640, 512, 1024, "fp16"),
    "max_segments_256": (8, 32, 64, 64, None, 0, 0, 0, "bf16"),
    "max_w_256_e1": (256, 1, 64, 128, None, 0, 0, 0, "bf16"),
    # The page's largest hidden and output sizes ("aclnnAlltoAllvGroupedMatMul",
    # Shape variables: H1, N1 < 65536; the shared expert's H2 <= 12288):
    # 512 K stages per tile with a K tail of 120, and 256 column tiles with a
    # ragged last one.
    "max_h1_65528": (2, 2, 65528, 136, [90, 130, 5, 70], 33, 12288, 72, "bf16"),
    "max_n1_65528": (2, 2, 64, 65528, [40, 3, 0, 90], 17, 64, 65528, "fp16"),
}


def edge_inputs(name, seed=1):
    W, e, H1, N1, rc, BS, H2, N2, dt = EDGE[name]
    if rc is None:
        from token_permute_grouped_gb300.workloads import random_counts
        rc = random_counts(W, e, 37 * W * e + 11, seed, 0.2)
    return custom_inputs(W, e, H1, N1, rc, dt, BS, H2, N2, seed=seed)


@pytest.mark.parametrize("want_perm", [True, False])
@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(orc, name, path, tiles, want_perm):
    # Without permuteOut the split path stages only the 128-row halves that
    # straddle a segment boundary and reads the others in place.
    inp = edge_inputs(name)
    gmmY, mmY, perm, (st, code) = run_gpu(inp, path, want_perm=want_perm, guard_rows=3, sentinel=0x7FC1,
                                          tiles=tiles)
    assert st == 0, code
    check_full(orc, inp, gmmY, mmY, perm)
    # Nothing written past the ends (guard rows keep the sentinel).
    for t, n in ((gmmY, inp.A), (perm, inp.A), (mmY, inp.wl.BS)):
        if t is not None:
            assert (t[n:].view(torch.int16) == 0x7FC1).all()


def _integer_inputs(W, e, H1, N1, rc, BS, H2, N2, dtype, seed):
    rng = np.random.default_rng(seed)
    A = int(np.sum(rc))
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    mk = lambda *s: torch.tensor(rng.integers(-4, 5, s), dtype=torch.float64).to(dt)
    base = custom_inputs(W, e, H1, N1, rc, dtype, BS, H2, N2)
    return Inputs(base.wl, np.asarray(rc, np.int32), mk(A, H1), mk(e, H1, N1),
                  mk(BS, H2) if BS else None, mk(H2, N2) if BS else None)


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_integer_inputs_bit_exact(orc, path, dtype, tiles):
    # |x|, |w| <= 4 and K <= 1024: every partial sum is an integer below 2^24,
    # exact in the fp32 accumulator in any order, so the output must be the
    # one nearest-even rounding of the exact (oracle) value.
    rc = [50, 0, 130, 7, 0, 260, 1, 90]
    inp = _integer_inputs(2, 4, 1024, 320, rc, 200, 512, 136, dtype, 3)
    gmmY, mmY, perm, (st, _) = run_gpu(inp, path, tiles=tiles)
    assert st == 0
    ref_perm, ref_y, ref_mm = orc.run(2, 4, inp.recvCounts, inp.ataOut, inp.gmmWeight, inp.mmX, inp.mmWeight)
    assert_bits_equal(perm, ref_perm, "permuteOut")
    assert_bits_equal(gmmY, rne_to(ref_y, inp.wl.torch_dtype), "gmmY")
    assert_bits_equal(mmY, rne_to(ref_mm, inp.wl.torch_dtype), "mmY")


@pytest.mark.parametrize("path", PATHS)
def test_identity_weight_reproduces_permute_out(orc, path):
    W, e, H = 4, 3, 256
    rc = [10, 200, 0, 3, 130, 1, 0, 0, 129, 64, 2, 5]
    base = custom_inputs(W, e, H, H, rc, "bf16")
    inp = Inputs(base.wl, base.recvCounts, base.ataOut, torch.eye(H).repeat(e, 1, 1).to(torch.bfloat16),
                 None, None)
    gmmY, _, perm, (st, _) = run_gpu(inp, path)
    assert st == 0
    assert_bits_equal(gmmY, perm, "gmmY vs permuteOut")
    assert_bits_equal(perm, orc.permute(W, e, inp.recvCounts, inp.ataOut), "permuteOut")


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("path", PATHS)
def test_deterministic(path, tiles):
    inp = edge_inputs("ragged_multi_tile", seed=4)
    a = run_gpu(inp, path, tiles=tiles)
    b = run_gpu(inp, path, tiles=tiles)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("want_perm", [True, False])
@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("path", PATHS)
def test_paths_agree_bitwise(path, tiles, want_perm):
    # Same fp32 accumulation order on every path and tile shape.
    inp = edge_inputs("fp16_mixed", seed=5)
    ref = run_gpu(inp, "split", tiles="single")
    got = run_gpu(inp, path, tiles=tiles, want_perm=want_perm)
    for x, y in zip(ref[:2], got[:2]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bad", ["sum_too_small", "negative"])
def test_device_detects_bad_counts(path, bad, tiles):
    inp = edge_inputs("ragged_multi_tile", seed=6)
    rc = inp.recvCounts.copy()
    big = int(np.argmax(rc))
    other = (big + 1) % len(rc)
    if bad == "sum_too_small":
        rc[big] -= 1
    else:
        rc[big] = -rc[big]
        rc[other] += 2 * inp.recvCounts[big]  # keeps the sum equal to A
    assert rc.sum() == inp.recvCounts.sum() - (bad == "sum_too_small")
    bad_inp = Inputs(inp.wl, rc, inp.ataOut, inp.gmmWeight, inp.mmX, inp.mmWeight)
    gmmY, mmY, perm, (st, code) = run_gpu(bad_inp, path, sentinel=0x1234, tiles=tiles)
    assert st == 6 and code & 1
    # Nothing written at all, shared expert included.
    for t in (gmmY, mmY, perm):
        assert (t.view(torch.int16) == 0x1234).all()
