"""a2av_gmm_run_static_scratch: the entry point that allocates nothing.

Some callers cannot allocate device memory: an operator embedded in a
framework or runtime that owns the device memory pool and hands it only its
inputs and outputs, or a latency-critical loop that must not call cudaMalloc
(it can block the host and synchronise the device).  For them the library
keeps a static scratch array in device memory and this entry point uses it
instead of a caller-provided workspace.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.  It passes alone in a fresh
process and after the other tests.  The static-scratch entry point runs the
same kernels on the same inputs as the workspace entry point
(a2av_gmm_run), so their outputs must agree bit for bit; the static-scratch
outputs are also checked against the oracle.  Two different problems run
back to back, so the second call finds the first call's leftovers in the
shared scratch array.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, check_full
from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import custom_inputs, random_counts

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
    cpu = lambda ts: tuple(None if t is None else t.cpu() for t in ts)
    return cpu(ref), cpu(got)


# Two problems run back to back through the same scratch array.  Without
# permuteOut the split path stages A * H1 * 2 bytes there (about 1.5 and
# 2.5 MiB), and split_runs stages only the 128-row halves that straddle a
# (source, expert) run boundary, so most of the second problem's staging
# area still holds the first problem's rows.  The split_runs shape has runs
# of several hundred rows, so it has halves read in place and staged ones.
CASES = {
    "split": [
        lambda: custom_inputs(4, 8, 512, 384, random_counts(4, 8, 1500, 3, 0.2), "bf16", 300, 320, 200, seed=3),
        lambda: custom_inputs(8, 4, 1024, 256, random_counts(8, 4, 1300, 4, 0.1), "fp16", 0, 0, 0, seed=4),
    ],
    "fused": [
        lambda: custom_inputs(4, 8, 512, 384, random_counts(4, 8, 1500, 3, 0.2), "bf16", 300, 320, 200, seed=3),
        lambda: custom_inputs(8, 4, 1024, 256, random_counts(8, 4, 1300, 4, 0.1), "fp16", 0, 0, 0, seed=4),
    ],
    "split_runs": [
        lambda: custom_inputs(8, 4, 1024, 256, random_counts(8, 4, 1300, 4, 0.1), "fp16", 0, 0, 0, seed=4),
        lambda: custom_inputs(2, 2, 512, 256, [700, 390, 45, 1010], "bf16", 130, 256, 128, seed=6),
    ],
}


@pytest.mark.parametrize("want_perm", [False, True])
@pytest.mark.parametrize("path", sorted(CASES))
def test_static_scratch_matches_workspace_entry_point_twice(orc, path, want_perm):
    assert torch.cuda.is_available(), "GPU test"
    build.build()
    for make in CASES[path]:
        inp = make()
        ref, got = _both(inp, path, want_perm)
        for name, r, g in zip(("gmmY", "mmY", "permuteOut"), ref, got):
            if r is not None:
                assert_bits_equal(g, r, name)
        check_full(orc, inp, got[0], got[1], got[2])


def test_static_scratch_rejects_oversized_problem():
    build.build()
    # Split path without permuteOut: A * H1 * 2 bytes of staging > 8 MiB.
    d = binding.make_desc(8, 4, 4096, 2048, 256, path="split")
    assert binding.a2av_gmm_workspace_size(d) > binding.STATIC_SCRATCH_BYTES
    p = 0x10000
    st = binding.load().a2av_gmm_run_static_scratch(
        binding.ctypes.byref(d), *[binding.ctypes.c_void_p(p)] * 8, None)
    assert binding.STATUS_NAMES[st] == "A2AV_ERR_SCRATCH_LIMIT"


# A child process without torch's CUDA state: it allocates through the CUDA
# runtime by ctypes, runs both entry points, resets the device
# (cudaDeviceReset ends this process's context; the module is loaded again
# afterwards), and runs both again.  The static-scratch call must find the
# array in the new context, not at its old address.
_CHILD = r"""
import ctypes, ctypes.util, json, sys
import numpy as np
import torch  # CPU tensors only: this process touches CUDA through the runtime below
sys.path.insert(0, sys.argv[1])
from token_permute_grouped_gb300 import binding
from token_permute_grouped_gb300.workloads import custom_inputs

def runtime():
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            pass
    return ctypes.CDLL("/usr/local/cuda/lib64/libcudart.so")

rt = runtime()
def ok(code, what):
    if code != 0:
        raise RuntimeError(f"{what}: CUDA error {code}")

def dev_copy(a):
    p = ctypes.c_void_p()
    ok(rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(max(a.nbytes, 16))), "cudaMalloc")
    ok(rt.cudaMemcpy(p, a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes), 1), "cudaMemcpy")
    return p

def dev_empty(nbytes):
    p = ctypes.c_void_p()
    ok(rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cudaMalloc")
    ok(rt.cudaMemset(p, 0x55, ctypes.c_size_t(nbytes)), "cudaMemset")
    return p

def host(p, shape):
    out = np.empty(shape, np.int16)
    ok(rt.cudaMemcpy(out.ctypes.data_as(ctypes.c_void_p), p, ctypes.c_size_t(out.nbytes), 2), "cudaMemcpy")
    return out

inp = custom_inputs(4, 2, 256, 128, [60, 0, 130, 70, 5, 200, 1, 90], "bf16", 70, 128, 64, seed=8)
wl = inp.wl
L = binding.load()
d = binding.make_desc(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, path="split")
ws_bytes = binding.a2av_gmm_workspace_size(d)
bits = lambda t: t.view(torch.int16).numpy()
arrays = [bits(inp.ataOut), inp.recvCounts.astype(np.int32), bits(inp.gmmWeight), bits(inp.mmX),
          bits(inp.mmWeight)]

def one_round():
    ata, rc, gw, mx, mw = (dev_copy(np.ascontiguousarray(a)) for a in arrays)
    res = {}
    for which in ("workspace", "static"):
        y = dev_empty(inp.A * wl.N1 * 2)
        m = dev_empty(wl.BS * wl.N2 * 2)
        if which == "workspace":
            ws = dev_empty(ws_bytes)
            st = L.a2av_gmm_run(ctypes.byref(d), ata, rc, gw, mx, mw, None, y, m, ws, ws_bytes, None)
        else:
            st = L.a2av_gmm_run_static_scratch(ctypes.byref(d), ata, rc, gw, mx, mw, None, y, m, None)
        if st != 0:
            raise RuntimeError(f"{which}: status {st}")
        ok(rt.cudaDeviceSynchronize(), "sync")
        res[which] = (host(y, (inp.A, wl.N1)), host(m, (wl.BS, wl.N2)))
    return res

first = one_round()
ok(rt.cudaDeviceReset(), "cudaDeviceReset")
second = one_round()
same = all(np.array_equal(a[k][i], b[k][i]) for a in (first, second) for b in (first, second)
           for k in ("workspace", "static") for i in (0, 1))
print(json.dumps({"bitwise_equal": bool(same)}))
"""


def test_static_scratch_after_device_reset():
    build.build()
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["bitwise_equal"], out
