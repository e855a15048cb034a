"""The debug build with device-side bounds checks (-DA2AV_CHECKS), on the GPU.

A failed check records kStatusBoundsCheck in the status word and skips the
access instead of trapping.  On consistent inputs no check may fire: the
checked build must report status 0 and give the same bits as the ordinary
build (the checks only read indices), and both must match the oracle
("aclnnAlltoAllvGroupedMatMul", Returns: a status code for every call).
"""

import ctypes

import pytest
import torch

from gpu_helpers import assert_bits_equal, check_full
from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import custom_inputs, random_counts

pytestmark = pytest.mark.gpu

CASES = {
    "ragged_multi_tile": lambda: custom_inputs(4, 8, 512, 384, random_counts(4, 8, 1500, 3, 0.2), "bf16",
                                               300, 320, 200, seed=3),
    "empty_groups_and_segments": lambda: custom_inputs(3, 5, 128, 96, [0, 5, 0, 129, 0, 0, 0, 0, 1, 0, 0, 7, 0, 128, 0],
                                                       "bf16", seed=2),
    "long_runs_fp16": lambda: custom_inputs(2, 2, 512, 256, [700, 390, 45, 1010], "fp16", 130, 256, 128, seed=6),
}


@pytest.fixture(scope="module")
def libs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build(checks=True)
    return binding.load(), binding.load_checks()


def _run(L, inp, path, want_perm):
    wl = inp.wl
    dev = torch.device("cuda:0")
    dt = wl.torch_dtype
    d = binding.make_desc(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, dt,
                          want_permute_out=want_perm, path=path)
    size = ctypes.c_size_t(0)
    assert L.a2av_gmm_workspace_size(ctypes.byref(d), ctypes.byref(size)) == 0
    ws = torch.empty(size.value, dtype=torch.uint8, device=dev)
    y = torch.empty(inp.A, wl.N1, dtype=dt, device=dev)
    m = torch.empty(wl.BS, wl.N2, dtype=dt, device=dev) if wl.BS else None
    perm = torch.empty(inp.A, wl.H1, dtype=dt, device=dev) if want_perm else None
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    ins = [inp.ataOut.to(dev), torch.from_numpy(inp.recvCounts).to(dev), inp.gmmWeight.to(dev),
           inp.mmX.to(dev) if wl.BS else None, inp.mmWeight.to(dev) if wl.BS else None]
    st = L.a2av_gmm_run(ctypes.byref(d), *[ptr(t) for t in ins], ptr(perm), ptr(y), ptr(m), ptr(ws), size.value,
                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    code = ctypes.c_int32(0)
    st = L.a2av_gmm_read_device_status(ptr(ws), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                       ctypes.byref(code))
    return st, code.value, y.cpu(), None if m is None else m.cpu(), None if perm is None else perm.cpu()


@pytest.mark.parametrize("want_perm", [False, True])
@pytest.mark.parametrize("path", ["fused", "split", "split_runs"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_checked_build_agrees_and_reports_nothing(orc, libs, name, path, want_perm):
    inp = CASES[name]()
    plain, checked = libs
    st, code, y, m, perm = _run(checked, inp, path, want_perm)
    assert (st, code) == (0, 0), (st, code)
    _, _, y0, m0, perm0 = _run(plain, inp, path, want_perm)
    assert_bits_equal(y, y0, "gmmY")
    if m is not None:
        assert_bits_equal(m, m0, "mmY")
    if perm is not None:
        assert_bits_equal(perm, perm0, "permuteOut")
    check_full(orc, inp, y, m, perm)


@pytest.mark.parametrize("i", range(0, 200, 5))
def test_checked_build_on_fuzz_shapes(orc, libs, i):
    # Forty of the seeded random shapes of test_gpu_fuzz.py, each on its drawn
    # path: no bounds check fires, and the bits equal the ordinary build's.
    from test_gpu_fuzz import _draw
    c = _draw(i)
    inp = custom_inputs(c["W"], c["e"], c["H1"], c["N1"], c["rc"], c["dtype"], c["BS"], c["H2"], c["N2"],
                        seed=c["seed"])
    plain, checked = libs
    st, code, y, m, perm = _run(checked, inp, c["path"], c["want_perm"])
    assert (st, code) == (0, 0), (c, st, code)
    _, _, y0, m0, perm0 = _run(plain, inp, c["path"], c["want_perm"])
    assert_bits_equal(y, y0, "gmmY")
    if m is not None:
        assert_bits_equal(m, m0, "mmY")
    if perm is not None:
        assert_bits_equal(perm, perm0, "permuteOut")
    check_full(orc, inp, y, m, perm)
