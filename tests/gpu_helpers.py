"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI binding and compare with the CPU oracle on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

from token_permute_grouped_gb300 import binding

TOL = 2e-2  # |gpu - ref| <= TOL * max(1, |ref|), against the float64 oracle


def run_gpu(inp, path="default", want_perm=True, guard_rows=0, sentinel=None, tiles="default"):
    """Run the hot path on cuda:0; returns CPU tensors (gmmY, mmY, permuteOut, status).

    With guard_rows, each output gets extra rows after its end, pre-filled with
    a sentinel pattern, so a test can check that nothing was written there.
    """
    wl = inp.wl
    dev = torch.device("cuda:0")
    dt = wl.torch_dtype
    plan = binding.Plan(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, dt,
                        want_permute_out=want_perm, path=path, device=dev, tiles=tiles)

    def out(rows, cols):
        t = torch.empty(rows + guard_rows, cols, dtype=dt, device=dev)
        t.view(torch.int16).fill_(sentinel if sentinel is not None else 0x7FC1)
        return t

    gmmY_full = out(inp.A, wl.N1)
    perm_full = out(inp.A, wl.H1) if want_perm else None
    mmY_full = out(wl.BS, wl.N2) if wl.BS else None
    rc = torch.from_numpy(inp.recvCounts).to(dev)
    mmX = inp.mmX.to(dev) if inp.mmX is not None else None
    mmW = inp.mmWeight.to(dev) if inp.mmWeight is not None else None
    plan.run(inp.ataOut.to(dev), rc, inp.gmmWeight.to(dev), mmX, mmW,
             gmmY=gmmY_full[:inp.A],
             mmY=mmY_full[:wl.BS] if mmY_full is not None else None,
             permuteOut=perm_full[:inp.A] if perm_full is not None else None)
    st, code = binding.a2av_gmm_read_device_status(plan.workspace)
    torch.cuda.synchronize()
    return (gmmY_full.cpu(), mmY_full.cpu() if mmY_full is not None else None,
            perm_full.cpu() if perm_full is not None else None, (st, code))


def assert_close(got: torch.Tensor, ref: np.ndarray, what: str):
    g = got.double().numpy()
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    err = np.abs(g - ref)
    lim = TOL * np.maximum(1.0, np.abs(ref))
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance, "
                             f"first {idx.tolist()}: got {g[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")


def assert_bits_equal(got: torch.Tensor, ref: torch.Tensor, what: str):
    a = got.contiguous().view(torch.int16)
    b = ref.contiguous().view(torch.int16)
    if not torch.equal(a, b):
        diff = (a != b).nonzero()
        raise AssertionError(f"{what}: {diff.shape[0]} elements differ, first {diff[:3].tolist()}")


def check_full(orc, inp, gmmY, mmY, perm):
    """Every element against the oracle."""
    wl = inp.wl
    ref_perm, ref_y, ref_mm = orc.run(wl.W, wl.e, inp.recvCounts, inp.ataOut, inp.gmmWeight, inp.mmX,
                                      inp.mmWeight)
    if perm is not None:
        assert_bits_equal(perm[:inp.A], ref_perm, "permuteOut")
    assert_close(gmmY[:inp.A], ref_y, "gmmY")
    if ref_mm is not None:
        assert_close(mmY[:wl.BS], ref_mm, "mmY")


def sample_rows(group_rows, n_random, seed, tile=128):
    """Rows worth checking: each group's first and last two rows, the rows on
    either side of each group's last tile boundary, and a seeded random set."""
    rows = set()
    start = 0
    A = int(np.sum(group_rows))
    for m in group_rows:
        m = int(m)
        if m:
            for r in (0, 1, m - 2, m - 1, (m - 1) // tile * tile, (m - 1) // tile * tile - 1):
                if 0 <= r < m:
                    rows.add(start + r)
        start += m
    if A:
        rng = np.random.default_rng(seed)
        rows.update(rng.integers(0, A, min(n_random, A)).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def rne_to(ref: np.ndarray, dtype) -> torch.Tensor:
    """Round float64 values to a 16-bit type.  Only used where the values are
    exactly representable in float32 (integer sums < 2^24), so the float64 ->
    float32 step is exact and the one rounding is float32 -> 16-bit, nearest
    even."""
    f32 = torch.from_numpy(ref.astype(np.float32))
    assert np.array_equal(f32.double().numpy(), ref)
    return f32.to(dtype)
