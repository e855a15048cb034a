"""The C ABI on the host: exports, phase-1 validation, phase-2 argument checks.

No GPU needed: every call here returns before the library touches CUDA.
"""

import ctypes
import glob
import os
import re
import subprocess

import pytest
import torch

from token_permute_grouped_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(a2av_\w+)\s*\(", text)))


def test_header_declares_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), name


def test_checks_build_exports_every_declared_symbol():
    # The debug build (-DA2AV_CHECKS: device-side bounds checks that record a
    # status bit) cross-compiles here and has the same C ABI.
    path = build.build(checks=True)
    assert path == build.CHECKS_LIB
    L = binding.load_checks()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.a2av_gmm_status_string(6).decode() == binding.load().a2av_gmm_status_string(6).decode()


def test_arrivals_argument_checks(lib):
    d = binding.make_desc(8, 4, 1000, 512, 256)
    args = [ctypes.c_void_p(0x10000 + 0x1000 * i) for i in range(8)]  # ataOut .. mmY
    ok_flags = ctypes.c_void_p(0x20000)
    call = lambda desc, flags: lib.a2av_gmm_run_arrivals(ctypes.byref(desc), *args, flags, ctypes.c_uint64(1),
                                                         ctypes.c_uint64(0), ctypes.c_void_p(0x40000),
                                                         ctypes.c_size_t(1 << 20), None)
    assert binding.STATUS_NAMES[call(d, None)] == "A2AV_ERR_NULLPTR"
    assert binding.STATUS_NAMES[call(d, ctypes.c_void_p(0x20004))] == "A2AV_ERR_UNSUPPORTED"  # not 8-byte aligned
    d_split = binding.make_desc(8, 4, 1000, 512, 256, path="split")
    assert binding.STATUS_NAMES[call(d_split, ok_flags)] == "A2AV_ERR_UNSUPPORTED"
    bad = binding.make_desc(8, 40, 1000, 512, 256)
    assert binding.STATUS_NAMES[call(bad, ok_flags)] == "A2AV_ERR_INVALID"


def ws(**kw):
    base = dict(W=8, e=4, A=16000, H1=4096, N1=1024, BS=2048, H2=4096, N2=1024)
    base.update(kw)
    d = binding.make_desc(**{k: base[k] for k in ("W", "e", "A", "H1", "N1", "BS", "H2", "N2")},
                          dtype=kw.get("dtype", torch.bfloat16), want_permute_out=kw.get("perm", False),
                          path=kw.get("path", "default"))
    for f in ("dtype", "tiles", "path"):
        if f"raw_{f}" in kw:
            setattr(d, f, kw[f"raw_{f}"])
    n = ctypes.c_size_t(0)
    st = binding.load().a2av_gmm_workspace_size(ctypes.byref(d), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"e": 32, "W": 8}, 0),
    ({"e": 33, "W": 1}, 2),             # e <= 32
    ({"e": 32, "W": 9}, 2),             # e * W <= 256
    ({"W": 0}, 2),
    ({"H1": 65536}, 2),                 # 0 < H1 < 65536
    ({"H1": 0}, 2),
    ({"N1": 65536}, 2),
    ({"H2": 12288}, 0),                 # 0 < H2 <= 12288
    ({"H2": 12296}, 2),
    ({"N2": 65536}, 2),
    ({"BS": 0, "H2": 0, "N2": 0}, 0),   # no shared expert
    ({"A": 0}, 0),                      # a rank may receive nothing
    ({"A": -1}, 2),
    ({"A": 2**31}, 2),
    ({"raw_dtype": 7}, 2),
    ({"raw_tiles": 4}, 2),
    ({"raw_tiles": 3}, 0),
    ({"raw_tiles": 2}, 0),
    ({"raw_path": 9}, 2),
    ({"raw_path": 3}, 0),
    ({"H1": 4100}, 3),                  # rows must start 16-byte aligned
    ({"N2": 1020}, 3),
    ({"dtype": torch.float16}, 0),
])
def test_phase1_validation(lib, kw, status):
    assert ws(**kw)[0] == status


def test_workspace_sizes(lib):
    assert ws(path="fused")[1] == 256
    assert ws(path="default", A=100, H1=64)[1] == 256 + 100 * 64 * 2  # default is the split path
    st, n = ws(path="split", A=1000, H1=512)
    assert st == 0 and n == 256 + 1000 * 512 * 2
    assert ws(path="split", A=1000, H1=512, perm=True)[1] == 256  # stages in permuteOut
    assert ws(path="split", A=0)[1] == 256


def test_launch_counts(lib):
    d = binding.make_desc(8, 4, 1000, 512, 256, path="fused")
    assert binding.a2av_gmm_launch_count(d) == 1
    d = binding.make_desc(8, 4, 1000, 512, 256)
    assert binding.a2av_gmm_launch_count(d) == 2
    d = binding.make_desc(8, 4, 1000, 512, 256, path="split")
    assert binding.a2av_gmm_launch_count(d) == 2
    d = binding.make_desc(8, 4, 0, 512, 256, path="split")
    assert binding.a2av_gmm_launch_count(d) == 1
    d = binding.make_desc(8, 40, 1000, 512, 256)
    assert binding.a2av_gmm_launch_count(d) == 0


def _run(lib, d, **ptrs):
    names = ["ataOut", "recvCounts", "gmmWeight", "mmX", "mmWeight", "permuteOut", "gmmY", "mmY", "workspace"]
    args = [ctypes.c_void_p(ptrs.get(n, 0x10000 + 0x1000 * i)) for i, n in enumerate(names)]
    return lib.a2av_gmm_run(ctypes.byref(d), *args, ptrs.get("wsbytes", 1 << 20), None)


def test_phase2_argument_checks(lib):
    d = binding.make_desc(8, 4, 1000, 512, 256, 64, 128, 64, want_permute_out=True)
    assert _run(lib, d, ataOut=0) == 1
    assert _run(lib, d, recvCounts=0) == 1
    assert _run(lib, d, gmmWeight=0) == 1
    assert _run(lib, d, mmX=0) == 1
    assert _run(lib, d, permuteOut=0) == 1
    assert _run(lib, d, workspace=0) == 1
    assert _run(lib, d, gmmY=0x10008) == 3        # not 16-byte aligned
    assert _run(lib, d, recvCounts=0x10002) == 3
    assert _run(lib, d, workspace=0x10080) == 4   # not 256-byte aligned
    assert _run(lib, d, wsbytes=100) == 4
    d.e = 99
    assert _run(lib, d) == 2
    # A = 0 and no shared expert: ataOut, gmmY, mmX... may all be NULL
    d = binding.make_desc(8, 4, 0, 512, 256, path="split")
    d2 = binding.make_desc(8, 4, 0, 512, 256, 64, 128, 64)
    assert _run(lib, d2, mmY=0) == 1


def qr(lib, W=8, rows=16, H=1024, qtype=0, mode=0, out_dtype=0, data=0x10000, scales=0x20000, out=0x30000):
    return lib.a2av_quant_reduce(W, rows, H, qtype, mode, ctypes.c_void_p(data), ctypes.c_void_p(scales),
                                 ctypes.c_void_p(out), out_dtype, None)


@pytest.mark.parametrize("kw,status", [
    ({"data": 0}, 1),
    ({"scales": 0}, 1),
    ({"out": 0}, 1),
    ({"W": 1}, 2), ({"W": 3}, 2), ({"W": 16}, 2),         # communicator size 2, 4 or 8
    ({"rows": 0}, 2),                                       # no empty tensors
    ({"H": 896}, 2), ({"H": 8320}, 2), ({"H": 1088}, 2),  # H in [1024, 8192], 128-aligned
    ({"qtype": 3}, 2), ({"qtype": -1}, 2),
    ({"mode": 2}, 2),
    ({"qtype": 2, "mode": 0}, 2),                           # mx quantisation takes FLOAT8 data only
    ({"out_dtype": 3}, 2),
    ({"data": 0x10008}, 3),                                 # data and out 16-byte aligned
    ({"out": 0x30004}, 3),
    ({"mode": 1, "scales": 0x20002}, 3),                    # float scales 4-byte aligned
])
def test_quant_reduce_argument_checks(lib, kw, status):
    assert qr(lib, **kw) == status


def mx_ws(**kw):
    base = dict(W=8, e=4, A=16000, H1=4096, N1=1024, BS=2048, H2=4096, N2=1024, qtype=0, want_permute_out=0,
                tiles=0)
    base.update(kw)
    d = binding.MxDesc(*(base[k] for k in ("W", "e", "A", "H1", "N1", "BS", "H2", "N2", "qtype",
                                            "want_permute_out", "tiles")))
    n = ctypes.c_size_t(0)
    return binding.load().a2av_gmm_mx_workspace_size(ctypes.byref(d), ctypes.byref(n)), n.value


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"qtype": 1}, 0),
    ({"qtype": 2}, 2),                  # E4M3FN or E5M2 codes only
    ({"e": 33}, 2),
    ({"W": 9, "e": 32}, 2),
    ({"H1": 65536}, 2),
    ({"H2": 12800}, 2),
    ({"A": -1}, 2),
    ({"H1": 4096 + 128}, 3),            # scale rows of H/32 bytes must be 16-byte multiples
    ({"H2": 1024 + 256}, 3),
    ({"N1": 1020}, 3),
    ({"BS": 0, "H2": 0, "N2": 0}, 0),
    ({"tiles": 1}, 0), ({"tiles": 2}, 0),
    ({"tiles": 3}, 2), ({"tiles": -1}, 2),  # default, single or pair
])
def test_mx_phase1_validation(lib, kw, status):
    assert mx_ws(**kw)[0] == status


def test_mx_workspace_sizes(lib):
    # Status word, staged codes (without permuteOut), then 512-byte scale
    # atoms, one per 128-row (or 128-column) block and per 128 codes of K:
    # routed A (an upper bound of ceil(A/128) + e halves), mmX, gmmWeight and
    # mmWeight; each part padded to 256 bytes.
    def atoms(blocks, K):
        return blocks * (K // 128) * 512
    routed = atoms(-(-1000 // 128) + 4, 512) + atoms(4 * (1024 // 128), 512)  # A = 1000, e = 4, N1 = 1024
    shared = atoms(2048 // 128, 4096) + atoms(1024 // 128, 4096)              # BS = 2048, N2 = 1024
    st, n = mx_ws(A=1000, H1=512)
    assert st == 0 and n == 256 + 512000 + routed + shared
    assert mx_ws(A=1000, H1=512, want_permute_out=1)[1] == 256 + routed + shared
    assert mx_ws(A=0)[1] == 256 + shared
    assert mx_ws(A=0, BS=0)[1] == 256


def test_status_strings(lib):
    for code in range(7):
        assert binding.a2av_gmm_status_string(code)
    assert "unknown" in binding.a2av_gmm_status_string(42)


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "nope.so"))
    with pytest.raises(ImportError):
        binding.load()
