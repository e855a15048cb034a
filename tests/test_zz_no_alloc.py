"""a2av_gmm_run_static_scratch: the entry point that allocates nothing.

Some callers cannot allocate device memory: an operator embedded in a
framework or runtime that owns the device memory pool and hands it only its
inputs and outputs, or a latency-critical loop that must not call cudaMalloc
(it can block the host and synchronise the device).  For them the library
keeps a static scratch array in device memory and this entry point uses it
instead of a caller-provided workspace.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.  It passes alone in a fresh
process and after the other tests.  Two calls in a row are checked against
the workspace entry point (a2av_gmm_run) within the parity tolerance the
other tests use; the second call finds the first call's leftovers in the
shared scratch array.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import TOL
from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import custom_inputs, random_counts

pytestmark = pytest.mark.gpu


def _both(inp, path, want_perm):
    """Outputs of the workspace entry point and of the static-scratch one."""
    wl = inp.wl
    dev = torch.device("cuda:0")
    dt = wl.torch_dtype
    d = binding.make_desc(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, dt,
                          want_permute_out=want_perm, path=path)
    ata = inp.ataOut.to(dev)
    rc = torch.from_numpy(inp.recvCounts).to(dev)
    gw = inp.gmmWeight.to(dev)
    mmX = inp.mmX.to(dev) if wl.BS else None
    mmW = inp.mmWeight.to(dev) if wl.BS else None

    def outputs():
        return (torch.full((inp.A, wl.N1), 7.0, dtype=dt, device=dev),
                torch.full((wl.BS, wl.N2), 7.0, dtype=dt, device=dev) if wl.BS else None,
                torch.full((inp.A, wl.H1), 7.0, dtype=dt, device=dev) if want_perm else None)

    ref = outputs()
    ws = torch.empty(binding.a2av_gmm_workspace_size(d), dtype=torch.uint8, device=dev)
    binding.a2av_gmm_run(d, ata, rc, gw, mmX, mmW, ref[2], ref[0], ref[1], ws)
    got = outputs()
    st = binding.a2av_gmm_run_static_scratch(d, ata, rc, gw, mmX, mmW, got[2], got[0], got[1])
    assert st == 0, binding.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    return ref, got


def _close(got, ref, what):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert np.all(np.abs(g - r) <= TOL * np.maximum(1.0, np.abs(r))), what


@pytest.mark.parametrize("path", ["split", "fused"])
def test_static_scratch_matches_workspace_entry_point_twice(path):
    assert torch.cuda.is_available(), "GPU test"
    build.build()
    # Two different problems back to back through the same scratch array;
    # the split path stages A * H1 * 2 bytes (about 1.5 and 2.5 MiB) in it.
    cases = [
        custom_inputs(4, 8, 512, 384, random_counts(4, 8, 1500, 3, 0.2), "bf16", 300, 320, 200, seed=3),
        custom_inputs(8, 4, 1024, 256, random_counts(8, 4, 1300, 4, 0.1), "fp16", 0, 0, 0, seed=4),
    ]
    for inp in cases:
        ref, got = _both(inp, path, want_perm=False)
        _close(got[0], ref[0], "gmmY")
        if ref[1] is not None:
            _close(got[1], ref[1], "mmY")


def test_static_scratch_rejects_oversized_problem():
    build.build()
    # Split path without permuteOut: A * H1 * 2 bytes of staging > 8 MiB.
    d = binding.make_desc(8, 4, 4096, 2048, 256, path="split")
    assert binding.a2av_gmm_workspace_size(d) > binding.STATIC_SCRATCH_BYTES
    p = 0x10000
    st = binding.load().a2av_gmm_run_static_scratch(
        binding.ctypes.byref(d), *[binding.ctypes.c_void_p(p)] * 8, None)
    assert binding.STATUS_NAMES[st] == "A2AV_ERR_SCRATCH_LIMIT"
