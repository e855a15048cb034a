"""The diagnostic entry points that time the grouped-GEMM kernel alone
(a2av_gmm_run_profiled, a2av_gmm_mx_run_profiled) on the GPU.

They do the same work as a2av_gmm_run / a2av_gmm_mx_run; only the launch of
the GEMM changes (plain stream order after the permute or prep kernel, with
two events around it).  So every output must be the same bits as the
ordinary call's, on every path and tile shape, and device-detected errors
must still reach the status word.  The events must bracket a positive time
no longer than the whole call's.
"""

import numpy as np
import pytest
import torch

from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import custom_inputs, make_mx_inputs, random_counts, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def _events():
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def _bits(t):
    return None if t is None else t.view(torch.int16).cpu()


@pytest.mark.parametrize("path,tiles", [("default", "default"), ("split", "single"), ("fused", "pair"),
                                        ("split_runs", "pair_k64")])
@pytest.mark.parametrize("want_perm", [False, True])
def test_bf16_same_bits_as_the_ordinary_call(path, tiles, want_perm):
    rc = random_counts(8, 4, 20000, seed=21, zero_prob=0.1)
    inp = custom_inputs(8, 4, 256, 512, rc, "bf16", 2048, 256, 384, seed=21)
    dev = torch.device("cuda:0")
    wl = inp.wl
    plan = binding.Plan(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, wl.torch_dtype, want_perm, path,
                        device=dev, tiles=tiles)
    args = (inp.ataOut.to(dev), torch.from_numpy(inp.recvCounts).to(dev), inp.gmmWeight.to(dev),
            inp.mmX.to(dev), inp.mmWeight.to(dev))
    start, end = _events()
    start.record()
    y, m, p = plan.run(*args)
    end.record()
    torch.cuda.synchronize()
    whole_ms = start.elapsed_time(end)
    ref = [_bits(t) for t in (y, m, p)]
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)
    ev = _events()
    y2, m2, p2 = plan.run(*args, gemm_events=ev)
    torch.cuda.synchronize()
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)
    for a, b, name in zip(ref, (y2, m2, p2), ("gmmY", "mmY", "permuteOut")):
        if a is not None:
            assert torch.equal(a, _bits(b)), name
    gemm_ms = ev[0].elapsed_time(ev[1])
    # The whole-call time above includes the first call's setup, so it bounds
    # the kernel alone from above with room to spare.
    assert 0.0 < gemm_ms <= whole_ms + 1.0, (gemm_ms, whole_ms)


def test_bf16_device_errors_still_reported():
    inp = custom_inputs(2, 2, 128, 128, [100, 50, 0, 80], "bf16", seed=22)
    dev = torch.device("cuda:0")
    wl = inp.wl
    plan = binding.Plan(wl.W, wl.e, inp.A, wl.H1, wl.N1, 0, 0, 0, wl.torch_dtype, False, "split", device=dev)
    bad = torch.from_numpy(np.array([100, 50, 0, 81], np.int32)).to(dev)  # sums to A + 1
    plan.run(inp.ataOut.to(dev), bad, inp.gmmWeight.to(dev), None, None, gemm_events=_events())
    torch.cuda.synchronize()
    st, code = binding.a2av_gmm_read_device_status(plan.workspace)
    assert binding.STATUS_NAMES[st] == "A2AV_ERR_DEVICE_CHECK" and code & 1, (st, code)
    # A good call on the same workspace clears the word again.
    plan.run(inp.ataOut.to(dev), torch.from_numpy(inp.recvCounts).to(dev), inp.gmmWeight.to(dev), None, None,
             gemm_events=_events())
    torch.cuda.synchronize()
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)


def _mx_case(seed=23):
    wl = Workload("mx_profiled", W=4, e=4, H1=1024, N1=512, dtype="bf16", routing="uniform",
                  BS=1024, H2=512, N2=256)
    rc = random_counts(4, 4, 12000, seed=seed, zero_prob=0.1)
    return make_mx_inputs(wl, seed=seed, recvCounts=np.asarray(rc, np.int32))


def _mx_run(plan, inp, recvCounts=None, gemm_events=None):
    dev = torch.device("cuda:0")
    d = lambda t: None if t is None else t.to(dev)
    rc = torch.from_numpy(inp.recvCounts if recvCounts is None else recvCounts).to(dev)
    out = plan.run(d(inp.ataOut_q), d(inp.ataOut_s), rc, d(inp.gmmWeight_q), d(inp.gmmWeight_s), d(inp.mmX_q),
                   d(inp.mmX_s), d(inp.mmWeight_q), d(inp.mmWeight_s), gemm_events=gemm_events)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("tiles", ["single", "pair"])
@pytest.mark.parametrize("want_perm", [False, True])
def test_mx_same_bits_as_the_ordinary_call(tiles, want_perm):
    inp = _mx_case()
    wl = inp.wl
    plan = binding.MxPlan(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, "e4m3fn", want_perm,
                          torch.device("cuda:0"), tiles)
    ref = [_bits(t) if t is not None and t.dtype == torch.bfloat16 else t for t in _mx_run(plan, inp)]
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)
    ev = _events()
    out = _mx_run(plan, inp, gemm_events=ev)
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)
    for a, b, name in zip(ref, out, ("gmmY", "mmY", "permuteOut_q", "permuteOut_s")):
        if a is None:
            assert b is None, name
        elif b.dtype == torch.bfloat16:
            assert torch.equal(a, _bits(b)), name
        else:
            assert torch.equal(a.cpu(), b.cpu()), name
    assert ev[0].elapsed_time(ev[1]) > 0.0


def test_mx_device_errors_still_reported():
    inp = _mx_case(seed=24)
    wl = inp.wl
    plan = binding.MxPlan(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, "e4m3fn", False,
                          torch.device("cuda:0"))
    bad = inp.recvCounts.copy()
    bad[-1] += 1  # sums to A + 1
    _mx_run(plan, inp, recvCounts=bad, gemm_events=_events())
    st, code = binding.a2av_gmm_read_device_status(plan.workspace)
    assert binding.STATUS_NAMES[st] == "A2AV_ERR_DEVICE_CHECK" and code & 1, (st, code)
    _mx_run(plan, inp, gemm_events=_events())
    assert binding.a2av_gmm_read_device_status(plan.workspace) == (0, 0)
