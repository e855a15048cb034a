"""Seeded random shapes on the GPU against the oracle, every element (needs a GB300).

"aclnnAlltoAllvGroupedMatMul", Shape variables: 1 <= e <= 32 local experts,
W * e <= 256 segments, H1 and N1 below 65536 (this library: multiples of 8),
the shared expert's H2 <= 12288; recvCounts any non-negative split of A,
empty segments and groups included.  Each case draws those within bounds
that keep the float64 oracle fast, picks a path and a tile shape, and checks
every output element (|gpu - ref| <= 2e-2 * max(1, |ref|); permuteOut bit
for bit).  The same inputs on the split path with single-CTA tiles must give
the same bits (every path and tile shape sums each output in the same
order).  The draws come from a fixed seed, so a failure names a case that
reproduces.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import check_full, run_gpu
from token_permute_grouped_gb300 import build
from token_permute_grouped_gb300.workloads import custom_inputs

pytestmark = pytest.mark.gpu

PATHS = ["default", "fused", "split", "split_runs"]
TILES = ["default", "single", "pair", "pair_k64"]
N_CASES = 200


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    e = int(rng.choice([1, 2, 3, 4, 7, 8, 16, 32]))
    W = int(rng.integers(1, max(2, min(9, 256 // e + 1))))
    H1 = int(rng.choice([8, 64, 72, 128, 200, 256, 520, 1024]))
    N1 = int(rng.choice([8, 16, 40, 64, 136, 256, 264, 640]))
    A = int(rng.integers(0, 3000))
    zero = float(rng.choice([0.0, 0.2, 0.6]))
    live = rng.random(W * e) >= zero
    w = rng.random(W * e) * live
    if A and w.sum() == 0:
        w[rng.integers(0, W * e)] = 1.0
    rc = np.zeros(W * e, np.int64) if A == 0 else np.floor(w / w.sum() * A).astype(np.int64)
    if A:
        rc[int(np.argmax(w))] += A - int(rc.sum())
    BS = int(rng.choice([0, 0, 1, 130, 700]))
    H2 = int(rng.choice([64, 136, 512])) if BS else 0
    N2 = int(rng.choice([8, 72, 256])) if BS else 0
    dtype = str(rng.choice(["bf16", "fp16"]))
    path = str(rng.choice(PATHS))
    tiles = str(rng.choice(TILES))
    want_perm = bool(rng.integers(0, 2))
    return dict(W=W, e=e, H1=H1, N1=N1, rc=rc.astype(np.int32), BS=BS, H2=H2, N2=N2, dtype=dtype, path=path,
                tiles=tiles, want_perm=want_perm, seed=1000 + i)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def test_draws_cover_the_bounds():
    cases = [_draw(i) for i in range(N_CASES)]
    assert all(c["W"] * c["e"] <= 256 and 1 <= c["e"] <= 32 for c in cases)
    assert any(c["rc"].sum() == 0 for c in cases) or any((c["rc"] == 0).any() for c in cases)
    assert {c["path"] for c in cases} == set(PATHS) and {c["tiles"] for c in cases} == set(TILES)
    assert {c["dtype"] for c in cases} == {"bf16", "fp16"}


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(orc, i):
    c = _draw(i)
    inp = custom_inputs(c["W"], c["e"], c["H1"], c["N1"], c["rc"], c["dtype"], c["BS"], c["H2"], c["N2"],
                        seed=c["seed"])
    gmmY, mmY, perm, (st, code) = run_gpu(inp, c["path"], want_perm=c["want_perm"], guard_rows=2, sentinel=0x7FC1,
                                          tiles=c["tiles"])
    assert st == 0, (c, code)
    check_full(orc, inp, gmmY, mmY, perm)
    for t, n in ((gmmY, inp.A), (perm, inp.A), (mmY, c["BS"])):
        if t is not None:
            assert (t[n:].view(torch.int16) == 0x7FC1).all(), ("written past the end", c)
    y0, m0, _, (st0, _) = run_gpu(inp, "split", want_perm=False, tiles="single")
    assert st0 == 0
    assert torch.equal(gmmY[:inp.A].view(torch.int16), y0[:inp.A].view(torch.int16)), c
    if c["BS"]:
        assert torch.equal(mmY[:c["BS"]].view(torch.int16), m0[:c["BS"]].view(torch.int16)), c


# ---- the block-scaled FP8 (mx) form: H1 and H2 multiples of 512, N1 and N2 of 8
N_MX = 60


def _draw_mx(i):
    rng = np.random.default_rng(5000 + i)
    e = int(rng.choice([1, 2, 4, 8, 32]))
    W = int(rng.integers(1, max(2, min(9, 256 // e + 1))))
    H1 = int(rng.choice([512, 1024, 1536, 2048]))
    N1 = int(rng.choice([8, 64, 136, 256, 392]))
    A = int(rng.integers(1, 1500))
    zero = float(rng.choice([0.0, 0.3]))
    live = rng.random(W * e) >= zero
    w = rng.random(W * e) * live
    if w.sum() == 0:
        w[rng.integers(0, W * e)] = 1.0
    rc = np.floor(w / w.sum() * A).astype(np.int64)
    rc[int(np.argmax(w))] += A - int(rc.sum())
    BS = int(rng.choice([0, 1, 257]))
    H2 = int(rng.choice([512, 1024])) if BS else 0
    N2 = int(rng.choice([8, 136])) if BS else 0
    return dict(W=W, e=e, H1=H1, N1=N1, rc=rc.astype(np.int32), BS=BS, H2=H2, N2=N2,
                qtype=str(rng.choice(["e4m3fn", "e5m2"])), tiles=str(rng.choice(["single", "pair"])),
                want_perm=bool(rng.integers(0, 2)), seed=5000 + i)


@pytest.mark.parametrize("i", range(N_MX))
def test_random_shape_mx(orc, i):
    from gpu_helpers import assert_close
    from token_permute_grouped_gb300 import binding
    from token_permute_grouped_gb300.workloads import Workload, make_mx_inputs
    c = _draw_mx(i)
    wl = Workload(f"mx_fuzz{i}", W=c["W"], e=c["e"], H1=c["H1"], N1=c["N1"], dtype="bf16", routing="given",
                  BS=c["BS"], H2=c["H2"], N2=c["N2"])
    inp = make_mx_inputs(wl, seed=c["seed"], qtype=c["qtype"], recvCounts=c["rc"])
    dev = torch.device("cuda:0")
    plan = binding.MxPlan(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, c["qtype"], c["want_perm"], dev,
                          c["tiles"])
    d = lambda t: None if t is None else t.to(dev)
    y, m, pq, ps = plan.run(d(inp.ataOut_q), d(inp.ataOut_s), torch.from_numpy(inp.recvCounts).to(dev),
                            d(inp.gmmWeight_q), d(inp.gmmWeight_s), d(inp.mmX_q), d(inp.mmX_s), d(inp.mmWeight_q),
                            d(inp.mmWeight_s))
    torch.cuda.synchronize()
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0), c
    q = {"e4m3fn": 0, "e5m2": 1}[c["qtype"]]
    perm_q = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut_q.view(torch.int16)).view(torch.uint8)
    perm_s = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut_s.view(torch.int16)).view(torch.uint8)
    if c["want_perm"]:
        assert torch.equal(pq.cpu(), perm_q) and torch.equal(ps.cpu(), perm_s), c
    _, _, groups, _ = orc.plan(wl.W, wl.e, inp.recvCounts, inp.A)
    ref = orc.mx_grouped_matmul(groups, perm_q, perm_s, inp.gmmWeight_q, inp.gmmWeight_s, q, q)
    assert_close(y.cpu(), ref, f"mx gmmY {c}")
    if wl.BS:
        ref_m = orc.mx_grouped_matmul([wl.BS], inp.mmX_q, inp.mmX_s, inp.mmWeight_q[None], inp.mmWeight_s[None], q, q)
        assert_close(m.cpu(), ref_m, f"mx mmY {c}")
