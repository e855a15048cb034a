"""CPU oracle for the AlltoAllv + Permute + GroupedMatMul hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``token_permute_grouped_gb300``) never does, and shares no code with it.

The arithmetic lives in ``a2av_ref.c`` (plain C, double accumulation, OpenMP
over output rows); this module builds it with gcc and wraps it with ctypes.
It follows the "Formula" section of the aclnnAlltoAllvGroupedMatMul page:
permuteOut = Permute(ataOut), gmmY = permuteOut x gmmWeight (one weight
matrix per local expert), mmY = mmX x mmWeight; the "Formula" of the
aclnnAmpUpdateScale page for the dynamic loss-scale update; and the
"Formula" and "Constraints" of the aclnnQuantReduceScatter page for the
dequantising reduce.

Every function is pinned by tests/test_oracle_pins.py; no function here is
"parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "a2av_ref.c")
_LIB = os.path.join(_HERE, "liba2av_ref.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {torch.bfloat16: 0, torch.float16: 1}


class OracleError(RuntimeError):
    pass


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (plain C11 + OpenMP)."""
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", *extra_flags,
           src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _declare(lib):
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.a2av_ref_decode.argtypes = [ctypes.c_int, p, i64, p]
    lib.a2av_ref_plan.argtypes = [i32, i32, p, i64, p, p, p, p]
    lib.a2av_ref_permute.argtypes = [i32, i32, p, i64, i64, p, p]
    lib.a2av_ref_grouped_matmul.argtypes = [i32, p, i64, i64, i64, i32, p, p, p, i64, p]
    lib.a2av_ref_matmul.argtypes = [i64, i64, i64, i32, p, p, p, i64, p]
    lib.a2av_ref_num_threads.argtypes = []
    lib.a2av_ref_set_threads.argtypes = [ctypes.c_int]
    lib.a2av_ref_amp_update_scale.argtypes = [p, p, ctypes.c_float, ctypes.c_float, ctypes.c_float, i32]
    lib.a2av_ref_any_nonfinite.argtypes = [ctypes.c_int, p, i64, p]
    lib.a2av_ref_decode8.argtypes = [ctypes.c_int, p, i64, p]
    lib.a2av_ref_quant_reduce.argtypes = [i32, i64, i64, i32, i32, p, p, p]
    lib.a2av_ref_mx_grouped_matmul.argtypes = [i32, p, i64, i64, i64, i32, i32, p, p, p, p, p, i64, p]
    for f in ("a2av_ref_decode", "a2av_ref_plan", "a2av_ref_permute",
              "a2av_ref_grouped_matmul", "a2av_ref_matmul", "a2av_ref_num_threads", "a2av_ref_set_threads",
              "a2av_ref_amp_update_scale", "a2av_ref_any_nonfinite", "a2av_ref_decode8",
              "a2av_ref_quant_reduce", "a2av_ref_mx_grouped_matmul"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def load_from(path: str):
    """Load an oracle build (tests use this for deliberately broken copies)."""
    return _declare(ctypes.CDLL(path))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB)
                    or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
                build()
            _lib = load_from(_LIB)
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        assert a.is_contiguous() and a.device.type == "cpu"
        return a.data_ptr()
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: oracle returned {rc}")


class Oracle:
    """Thin wrapper; ``impl`` lets tests swap in a deliberately broken build."""

    def __init__(self, impl=None):
        self.L = impl if impl is not None else lib()

    def num_threads(self) -> int:
        return int(self.L.a2av_ref_num_threads())

    def set_threads(self, n: int) -> int:
        """OpenMP threads for the following calls (results do not depend on it)."""
        return int(self.L.a2av_ref_set_threads(n))

    def decode(self, t: torch.Tensor) -> np.ndarray:
        b = _bits(t).reshape(-1)
        out = np.empty(b.numel(), dtype=np.float64)
        _check(self.L.a2av_ref_decode(DTYPE_CODE[t.dtype], _ptr(b), b.numel(), _ptr(out)), "decode")
        return out.reshape(tuple(t.shape))

    def plan(self, W: int, e: int, recvCounts, A: int):
        rc = np.ascontiguousarray(recvCounts, dtype=np.int32)
        E = W * e
        src = np.zeros(E, np.int64)
        dst = np.zeros(E, np.int64)
        gr = np.zeros(e, np.int64)
        go = np.zeros(e + 1, np.int64)
        _check(self.L.a2av_ref_plan(W, e, _ptr(rc), A, _ptr(src), _ptr(dst), _ptr(gr), _ptr(go)), "plan")
        return src, dst, gr, go

    def permute(self, W: int, e: int, recvCounts, ataOut: torch.Tensor) -> torch.Tensor:
        rc = np.ascontiguousarray(recvCounts, dtype=np.int32)
        A, H1 = ataOut.shape
        out = torch.empty_like(ataOut)
        _check(self.L.a2av_ref_permute(W, e, _ptr(rc), A, H1, _ptr(_bits(ataOut)),
                                       _ptr(out.view(torch.int16))), "permute")
        return out

    def grouped_matmul(self, group_rows, permuteOut: torch.Tensor, gmmWeight: torch.Tensor,
                       rows=None) -> np.ndarray:
        gr = np.ascontiguousarray(group_rows, dtype=np.int64)
        e, H1, N1 = gmmWeight.shape
        A = permuteOut.shape[0]
        assert permuteOut.shape[1] == H1 and permuteOut.dtype == gmmWeight.dtype
        rl = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = A if rl is None else len(rl)
        out = np.empty((n, N1), np.float64)
        _check(self.L.a2av_ref_grouped_matmul(
            e, _ptr(gr), A, H1, N1, DTYPE_CODE[gmmWeight.dtype], _ptr(_bits(permuteOut)),
            _ptr(_bits(gmmWeight)), _ptr(rl), n, _ptr(out)), "grouped_matmul")
        return out

    def matmul(self, mmX: torch.Tensor, mmWeight: torch.Tensor, rows=None) -> np.ndarray:
        BS, H2 = mmX.shape
        H2b, N2 = mmWeight.shape
        assert H2 == H2b and mmX.dtype == mmWeight.dtype
        rl = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = BS if rl is None else len(rl)
        out = np.empty((n, N2), np.float64)
        _check(self.L.a2av_ref_matmul(BS, H2, N2, DTYPE_CODE[mmX.dtype], _ptr(_bits(mmX)),
                                      _ptr(_bits(mmWeight)), _ptr(rl), n, _ptr(out)), "matmul")
        return out

    def amp_update_scale(self, scale: float, growth_tracker: int, found_inf: float, growth_factor: float,
                         backoff_factor: float, growth_interval: int):
        """Page "aclnnAmpUpdateScale": returns (updated_scale, updated_tracker), float32 arithmetic."""
        sc = ctypes.c_float(scale)
        tr = ctypes.c_int32(growth_tracker)
        _check(self.L.a2av_ref_amp_update_scale(ctypes.byref(sc), ctypes.byref(tr), found_inf, growth_factor,
                                                backoff_factor, growth_interval), "amp_update_scale")
        return sc.value, tr.value

    def any_nonfinite(self, t: torch.Tensor) -> bool:
        code = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}[t.dtype]
        b = t.contiguous().reshape(-1)
        found = ctypes.c_int32(0)
        _check(self.L.a2av_ref_any_nonfinite(code, b.data_ptr() if b.numel() else None, b.numel(),
                                             ctypes.byref(found)), "any_nonfinite")
        return bool(found.value)

    def decode8(self, kind: int, bits: np.ndarray) -> np.ndarray:
        """kind 0 E4M3FN, 1 E5M2, 2 INT8, 3 E8M0 (bytes as uint8)."""
        b = np.ascontiguousarray(bits, dtype=np.uint8)
        out = np.empty(b.size, np.float64)
        _check(self.L.a2av_ref_decode8(kind, _ptr(b) if b.size else None, b.size, _ptr(out)), "decode8")
        return out.reshape(b.shape)

    def quant_reduce(self, data: np.ndarray, scales: np.ndarray, qtype: int, mode: int) -> np.ndarray:
        """Page "aclnnQuantReduceScatter": data [W, rows, H] uint8, scales [W, rows, H/32] uint8
        (mode 0, E8M0) or [W, rows, H/128] float32 (mode 1); returns [rows, H] float64."""
        W, rows, H = data.shape
        d = np.ascontiguousarray(data, dtype=np.uint8)
        sc = np.ascontiguousarray(scales)
        out = np.empty((rows, H), np.float64)
        _check(self.L.a2av_ref_quant_reduce(W, rows, H, qtype, mode, _ptr(d), _ptr(sc), _ptr(out)),
               "quant_reduce")
        return out

    def mx_grouped_matmul(self, group_rows, a, sa, w, sw, qa: int, qw: int, rows=None) -> np.ndarray:
        """Block-scaled FP8 grouped product: a [A, K] codes, sa [A, K/32] E8M0, w [e, N, K]
        codes, sw [e, N, K/32] E8M0 (all uint8); qa, qw 0 = E4M3FN, 1 = E5M2.  Returns
        [len(rows) or A, N] float64.  A shared-expert product is the case e = 1."""
        gr = np.ascontiguousarray(group_rows, dtype=np.int64)
        a, sa, w, sw = (np.ascontiguousarray(t.numpy() if isinstance(t, torch.Tensor) else t, dtype=np.uint8)
                        for t in (a, sa, w, sw))
        A, K = a.shape
        e, N, K2 = w.shape
        assert K2 == K and sa.shape == (A, K // 32) and sw.shape == (e, N, K // 32) and len(gr) == e
        rl = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = A if rl is None else len(rl)
        out = np.empty((n, N), np.float64)
        _check(self.L.a2av_ref_mx_grouped_matmul(e, _ptr(gr), A, K, N, qa, qw, _ptr(a), _ptr(sa), _ptr(w),
                                                 _ptr(sw), _ptr(rl), 0 if rl is None else n, _ptr(out)),
               "mx_grouped_matmul")
        return out

    def run(self, W: int, e: int, recvCounts, ataOut, gmmWeight, mmX=None, mmWeight=None,
            gmm_rows=None, mm_rows=None):
        """The whole hot path: (permuteOut, gmmY rows, mmY rows or None)."""
        perm = self.permute(W, e, recvCounts, ataOut)
        _, _, gr, _ = self.plan(W, e, recvCounts, ataOut.shape[0])
        gmmY = self.grouped_matmul(gr, perm, gmmWeight, gmm_rows)
        mmY = None
        if mmX is not None:
            mmY = self.matmul(mmX, mmWeight, mm_rows)
        return perm, gmmY, mmY
