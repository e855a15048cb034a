"""ctypes binding of liba2av_gmm.so: argument marshalling only.

Same names as the C ABI in include/a2av_gmm.h.  Every step of the hot path
runs in the library's CUDA kernels; this module only checks tensors, sizes the
outputs and workspace with torch, and passes raw device pointers and the
current CUDA stream.  There is no CPU fallback: without the built library
every entry point raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

A2AV_OK = 0
STATUS_NAMES = {0: "A2AV_OK", 1: "A2AV_ERR_NULLPTR", 2: "A2AV_ERR_INVALID", 3: "A2AV_ERR_UNSUPPORTED",
                4: "A2AV_ERR_WORKSPACE", 5: "A2AV_ERR_CUDA", 6: "A2AV_ERR_DEVICE_CHECK",
                7: "A2AV_ERR_SCRATCH_LIMIT", 8: "A2AV_ERR_ARRIVAL_TIMEOUT"}
STATIC_SCRATCH_BYTES = 256 + (8 << 20)  # A2AV_STATIC_SCRATCH_BYTES
DTYPES = {torch.bfloat16: 0, torch.float16: 1}
PATHS = {"default": 0, "fused": 1, "split": 2, "split_runs": 3}
TILES = {"default": 0, "single": 1, "pair": 2, "pair_k64": 3}

# Every function the headers under include/ declare.
EXPORTS = ("a2av_gmm_workspace_size", "a2av_gmm_run", "a2av_gmm_read_device_status",
           "a2av_gmm_status_string", "a2av_gmm_launch_count", "a2av_gmm_run_static_scratch",
           "a2av_gmm_run_profiled", "a2av_gmm_run_arrivals",
           "a2av_amp_update_scale", "a2av_found_nonfinite", "a2av_quant_reduce",
           "a2av_gmm_mx_workspace_size", "a2av_gmm_mx_run", "a2av_gmm_mx_run_profiled")

# a2av_qtype / a2av_qmode of include/a2av_quant_reduce.h.
QTYPES = {"e4m3fn": 0, "e5m2": 1, "int8": 2}
QMODES = {"mx": 0, "group128": 1}


class A2avError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [("W", ctypes.c_int32), ("e", ctypes.c_int32),
                ("A", ctypes.c_int64), ("H1", ctypes.c_int64), ("N1", ctypes.c_int64),
                ("BS", ctypes.c_int64), ("H2", ctypes.c_int64), ("N2", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("want_permute_out", ctypes.c_int32),
                ("path", ctypes.c_int32), ("tiles", ctypes.c_int32)]


class MxDesc(ctypes.Structure):
    """a2av_gmm_mx_desc of include/a2av_gmm_mx.h."""
    _fields_ = [("W", ctypes.c_int32), ("e", ctypes.c_int32),
                ("A", ctypes.c_int64), ("H1", ctypes.c_int64), ("N1", ctypes.c_int64),
                ("BS", ctypes.c_int64), ("H2", ctypes.c_int64), ("N2", ctypes.c_int64),
                ("qtype", ctypes.c_int32), ("want_permute_out", ctypes.c_int32), ("tiles", ctypes.c_int32)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load():
    """Load the built library (raises if it was not built)."""
    global _lib
    if _lib is None:
        _lib = load_library(_build.LIB)
    return _lib


def load_checks():
    """The debug build with device-side bounds checks (built by build.build(checks=True)),
    as a separate handle with the same functions."""
    return load_library(_build.CHECKS_LIB)


def load_library(path: str):
    """Open one build of the library and declare every C-ABI function's signature."""
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} (run __graft_entry__.build())")
    L = ctypes.CDLL(path)
    p, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    L.a2av_gmm_workspace_size.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(sz)]
    L.a2av_gmm_workspace_size.restype = ctypes.c_int
    L.a2av_gmm_run.argtypes = [ctypes.POINTER(Desc), p, p, p, p, p, p, p, p, p, sz, p]
    L.a2av_gmm_run.restype = ctypes.c_int
    L.a2av_gmm_run_profiled.argtypes = [ctypes.POINTER(Desc), p, p, p, p, p, p, p, p, p, sz, p, p, p]
    L.a2av_gmm_run_profiled.restype = ctypes.c_int
    L.a2av_gmm_run_arrivals.argtypes = [ctypes.POINTER(Desc), p, p, p, p, p, p, p, p, p, ctypes.c_uint64,
                                        ctypes.c_uint64, p, sz, p]
    L.a2av_gmm_run_arrivals.restype = ctypes.c_int
    L.a2av_gmm_read_device_status.argtypes = [p, p, ctypes.POINTER(i32)]
    L.a2av_gmm_read_device_status.restype = ctypes.c_int
    L.a2av_gmm_status_string.argtypes = [ctypes.c_int]
    L.a2av_gmm_status_string.restype = ctypes.c_char_p
    L.a2av_gmm_launch_count.argtypes = [ctypes.POINTER(Desc)]
    L.a2av_gmm_launch_count.restype = i32
    L.a2av_gmm_run_static_scratch.argtypes = [ctypes.POINTER(Desc), p, p, p, p, p, p, p, p, p]
    L.a2av_gmm_run_static_scratch.restype = ctypes.c_int
    L.a2av_amp_update_scale.argtypes = [p, p, p, ctypes.c_float, ctypes.c_float, i32, p]
    L.a2av_amp_update_scale.restype = ctypes.c_int
    L.a2av_found_nonfinite.argtypes = [p, ctypes.c_int64, i32, p, p]
    L.a2av_found_nonfinite.restype = ctypes.c_int
    L.a2av_quant_reduce.argtypes = [i32, ctypes.c_int64, ctypes.c_int64, i32, i32, p, p, p, i32, p]
    L.a2av_quant_reduce.restype = ctypes.c_int
    L.a2av_gmm_mx_workspace_size.argtypes = [ctypes.POINTER(MxDesc), ctypes.POINTER(sz)]
    L.a2av_gmm_mx_workspace_size.restype = ctypes.c_int
    L.a2av_gmm_mx_run.argtypes = [ctypes.POINTER(MxDesc)] + [p] * 14 + [sz, p]
    L.a2av_gmm_mx_run.restype = ctypes.c_int
    L.a2av_gmm_mx_run_profiled.argtypes = [ctypes.POINTER(MxDesc)] + [p] * 14 + [sz, p, p, p]
    L.a2av_gmm_mx_run_profiled.restype = ctypes.c_int
    return L


def make_desc(W, e, A, H1, N1, BS=0, H2=0, N2=0, dtype=torch.bfloat16, want_permute_out=False,
              path="default", tiles="default") -> Desc:
    return Desc(W, e, A, H1, N1, BS, H2, N2, DTYPES[dtype], int(bool(want_permute_out)), PATHS[path],
                TILES[tiles])


def a2av_gmm_workspace_size(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    st = load().a2av_gmm_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    if st != A2AV_OK:
        raise A2avError(st, "a2av_gmm_workspace_size")
    return n.value


def a2av_gmm_launch_count(desc: Desc) -> int:
    return int(load().a2av_gmm_launch_count(ctypes.byref(desc)))


def a2av_gmm_status_string(status: int) -> str:
    return load().a2av_gmm_status_string(status).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def a2av_gmm_run(desc: Desc, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY, mmY,
                 workspace: torch.Tensor, stream=None) -> None:
    """Raw phase 2: device tensors (or None) in, enqueued on the stream."""
    s = stream if stream is not None else torch.cuda.current_stream()
    st = load().a2av_gmm_run(ctypes.byref(desc), _ptr(ataOut), _ptr(recvCounts), _ptr(gmmWeight),
                             _ptr(mmX), _ptr(mmWeight), _ptr(permuteOut), _ptr(gmmY), _ptr(mmY),
                             _ptr(workspace), workspace.numel(), ctypes.c_void_p(s.cuda_stream))
    if st != A2AV_OK:
        raise A2avError(st, "a2av_gmm_run")


def a2av_gmm_run_profiled(desc: Desc, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY, mmY,
                          workspace: torch.Tensor, gemm_begin: torch.cuda.Event, gemm_end: torch.cuda.Event,
                          stream=None) -> None:
    """a2av_gmm_run with two timing events (torch.cuda.Event(enable_timing=True)) recorded
    right before and after the grouped-GEMM kernel."""
    s = stream if stream is not None else torch.cuda.current_stream()
    for ev in (gemm_begin, gemm_end):
        if ev.cuda_event == 0:  # created lazily by torch: make it exist on this device
            ev.record(s)
    st = load().a2av_gmm_run_profiled(ctypes.byref(desc), _ptr(ataOut), _ptr(recvCounts), _ptr(gmmWeight),
                                      _ptr(mmX), _ptr(mmWeight), _ptr(permuteOut), _ptr(gmmY), _ptr(mmY),
                                      _ptr(workspace), workspace.numel(), ctypes.c_void_p(s.cuda_stream),
                                      ctypes.c_void_p(gemm_begin.cuda_event), ctypes.c_void_p(gemm_end.cuda_event))
    if st != A2AV_OK:
        raise A2avError(st, "a2av_gmm_run_profiled")


def a2av_gmm_run_arrivals(desc: Desc, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY, mmY,
                          arrived: torch.Tensor, arrival_tag: int, wait_limit_ns: int, workspace: torch.Tensor,
                          stream=None) -> None:
    """a2av_gmm_run that starts before the rows have all arrived: source w's rows of ataOut are
    read once arrived[w] (an int64 device tensor of W flags) equals arrival_tag."""
    _check(arrived, "arrived", torch.int64, 1)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = load().a2av_gmm_run_arrivals(ctypes.byref(desc), _ptr(ataOut), _ptr(recvCounts), _ptr(gmmWeight),
                                      _ptr(mmX), _ptr(mmWeight), _ptr(permuteOut), _ptr(gmmY), _ptr(mmY),
                                      _ptr(arrived), ctypes.c_uint64(arrival_tag & (2**64 - 1)),
                                      ctypes.c_uint64(wait_limit_ns), _ptr(workspace), workspace.numel(),
                                      ctypes.c_void_p(s.cuda_stream))
    if st != A2AV_OK:
        raise A2avError(st, "a2av_gmm_run_arrivals")


def a2av_gmm_run_static_scratch(desc: Desc, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY,
                                mmY, stream=None) -> int:
    """Phase 2 without a workspace, for callers that cannot allocate device
    memory: the library's own static device scratch array stands in for it.
    Returns the status code (0 = enqueued)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load().a2av_gmm_run_static_scratch(
        ctypes.byref(desc), _ptr(ataOut), _ptr(recvCounts), _ptr(gmmWeight), _ptr(mmX), _ptr(mmWeight),
        _ptr(permuteOut), _ptr(gmmY), _ptr(mmY), ctypes.c_void_p(s.cuda_stream)))


def a2av_amp_update_scale(scale: torch.Tensor, growth_tracker: torch.Tensor, found_inf: torch.Tensor,
                          growth_factor: float, backoff_factor: float, growth_interval: int, stream=None) -> None:
    """In place on device scalars: scale (float32 [1]), growth_tracker (int32 [1]), found_inf (float32 [1])."""
    _check(scale, "scale", torch.float32)
    _check(growth_tracker, "growth_tracker", torch.int32)
    _check(found_inf, "found_inf", torch.float32)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = load().a2av_amp_update_scale(_ptr(scale), _ptr(growth_tracker), _ptr(found_inf), growth_factor,
                                      backoff_factor, growth_interval, ctypes.c_void_p(s.cuda_stream))
    if st != A2AV_OK:
        raise A2avError(st, "a2av_amp_update_scale")


def a2av_found_nonfinite(x: torch.Tensor, found_inf: torch.Tensor, stream=None) -> None:
    """found_inf (float32 [1], device) = 1 when x holds an inf or NaN; unchanged otherwise."""
    code = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}[x.dtype]
    _check(x, "x")
    _check(found_inf, "found_inf", torch.float32)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = load().a2av_found_nonfinite(_ptr(x) if x.numel() else None, x.numel(), code, _ptr(found_inf),
                                     ctypes.c_void_p(s.cuda_stream))
    if st != A2AV_OK:
        raise A2avError(st, "a2av_found_nonfinite")


def a2av_quant_reduce(data: torch.Tensor, scales: torch.Tensor, qtype: str, mode: str,
                      out: torch.Tensor, stream=None) -> torch.Tensor:
    """out [rows, H] = sum over w of decode(data[w]) * scales[w] ("aclnnQuantReduceScatter" page,
    Formula).  data: uint8 [W, rows, H] codes of qtype ("e4m3fn", "e5m2", "int8"); scales: uint8
    E8M0 [W, rows, H/32] for mode "mx", float32 [W, rows, H/128] for "group128"; out: bf16, fp16
    or fp32 [rows, H]."""
    _check(data, "data", torch.uint8, 3)
    _check(scales, "scales", torch.uint8 if mode == "mx" else torch.float32, 3)
    _check(out, "out", None, 2)
    W, rows, H = data.shape
    if tuple(out.shape) != (rows, H):
        raise ValueError(f"out must be [{rows}, {H}], got {tuple(out.shape)}")
    code = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}[out.dtype]
    s = stream if stream is not None else torch.cuda.current_stream()
    st = load().a2av_quant_reduce(W, rows, H, QTYPES[qtype], QMODES[mode], _ptr(data), _ptr(scales),
                                  _ptr(out), code, ctypes.c_void_p(s.cuda_stream))
    if st != A2AV_OK:
        raise A2avError(st, "a2av_quant_reduce")
    return out


def a2av_gmm_read_device_status(workspace: torch.Tensor, stream=None) -> tuple[int, int]:
    s = stream if stream is not None else torch.cuda.current_stream()
    code = ctypes.c_int32(0)
    st = load().a2av_gmm_read_device_status(_ptr(workspace), ctypes.c_void_p(s.cuda_stream),
                                             ctypes.byref(code))
    return st, code.value


def _check(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


class Plan:
    """Descriptor + workspace for one shape, reusable across calls."""

    def __init__(self, W, e, A, H1, N1, BS=0, H2=0, N2=0, dtype=torch.bfloat16,
                 want_permute_out=False, path="default", device=None, tiles="default"):
        self.desc = make_desc(W, e, A, H1, N1, BS, H2, N2, dtype, want_permute_out, path, tiles)
        self.dtype = dtype
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.workspace = torch.empty(a2av_gmm_workspace_size(self.desc), dtype=torch.uint8, device=self.device)

    def run(self, ataOut, recvCounts, gmmWeight, mmX=None, mmWeight=None, gmmY=None, mmY=None,
            permuteOut=None, stream=None, gemm_events=None):
        """gemm_events: optional (begin, end) timing events recorded around the GEMM kernel
        (a2av_gmm_run_profiled)."""
        d = self.desc
        if d.A:
            _check(ataOut, "ataOut", self.dtype, 2)
        _check(recvCounts, "recvCounts", torch.int32, 1)
        _check(gmmWeight, "gmmWeight", self.dtype, 3)
        if tuple(gmmWeight.shape) != (d.e, d.H1, d.N1):
            raise ValueError("gmmWeight shape")
        if recvCounts.numel() != d.W * d.e:
            raise ValueError("recvCounts length")
        if gmmY is None:
            gmmY = torch.empty(d.A, d.N1, dtype=self.dtype, device=self.device)
        if d.want_permute_out and permuteOut is None:
            permuteOut = torch.empty(d.A, d.H1, dtype=self.dtype, device=self.device)
        if d.BS:
            _check(mmX, "mmX", self.dtype, 2)
            _check(mmWeight, "mmWeight", self.dtype, 2)
            if mmY is None:
                mmY = torch.empty(d.BS, d.N2, dtype=self.dtype, device=self.device)
        args = (d, ataOut if d.A else None, recvCounts, gmmWeight, mmX, mmWeight,
                permuteOut if d.want_permute_out else None, gmmY if d.A else None,
                mmY if d.BS else None, self.workspace)
        if gemm_events is None:
            a2av_gmm_run(*args, stream)
        else:
            a2av_gmm_run_profiled(*args, gemm_events[0], gemm_events[1], stream)
        return gmmY, mmY, permuteOut


def a2av_gmm(ataOut, recvCounts, gmmWeight, mmX=None, mmWeight=None, return_permute=False,
             W=None, path="default", tiles="default"):
    """permuteOut = Permute(ataOut); gmmY = permuteOut x gmmWeight; mmY = mmX x mmWeight.

    Returns (gmmY, mmY or None, permuteOut or None).  W defaults to
    len(recvCounts) // e.
    """
    e, H1, N1 = gmmWeight.shape
    if W is None:
        W = recvCounts.numel() // e
    BS, H2, N2 = (0, 0, 0)
    if mmX is not None:
        BS, H2 = mmX.shape
        N2 = mmWeight.shape[1]
    plan = Plan(W, e, ataOut.shape[0], H1, N1, BS, H2, N2, gmmWeight.dtype, return_permute, path,
                device=gmmWeight.device, tiles=tiles)
    return plan.run(ataOut, recvCounts, gmmWeight, mmX, mmWeight)


class MxPlan:
    """Descriptor + workspace of the block-scaled FP8 (mx) call for one shape
    (include/a2av_gmm_mx.h): codes as uint8 tensors, E8M0 scales as uint8
    tensors with one byte per 32 codes along K, weights [e, N1, H1]."""

    def __init__(self, W, e, A, H1, N1, BS=0, H2=0, N2=0, qtype="e4m3fn", want_permute_out=False, device=None,
                 tiles="default"):
        self.desc = MxDesc(W, e, A, H1, N1, BS, H2, N2, QTYPES[qtype], int(bool(want_permute_out)), TILES[tiles])
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        n = ctypes.c_size_t(0)
        st = load().a2av_gmm_mx_workspace_size(ctypes.byref(self.desc), ctypes.byref(n))
        if st != A2AV_OK:
            raise A2avError(st, "a2av_gmm_mx_workspace_size")
        self.workspace = torch.empty(n.value, dtype=torch.uint8, device=self.device)

    def run(self, ataOut_q, ataOut_s, recvCounts, gmmWeight_q, gmmWeight_s, mmX_q=None, mmX_s=None,
            mmWeight_q=None, mmWeight_s=None, gmmY=None, mmY=None, permuteOut_q=None, permuteOut_s=None,
            stream=None, gemm_events=None):
        """Returns (gmmY, mmY, permuteOut_q, permuteOut_s); outputs are bf16.
        gemm_events: optional (begin, end) timing events recorded around the
        GEMM kernel (a2av_gmm_mx_run_profiled)."""
        d = self.desc
        for t, name in ((ataOut_q, "ataOut_q"), (ataOut_s, "ataOut_s")):
            if d.A:
                _check(t, name, torch.uint8, 2)
        _check(recvCounts, "recvCounts", torch.int32, 1)
        _check(gmmWeight_q, "gmmWeight_q", torch.uint8, 3)
        _check(gmmWeight_s, "gmmWeight_s", torch.uint8, 3)
        if tuple(gmmWeight_q.shape) != (d.e, d.N1, d.H1) or tuple(gmmWeight_s.shape) != (d.e, d.N1, d.H1 // 32):
            raise ValueError("gmmWeight_q must be [e, N1, H1] and gmmWeight_s [e, N1, H1/32]")
        if d.A and (tuple(ataOut_q.shape) != (d.A, d.H1) or tuple(ataOut_s.shape) != (d.A, d.H1 // 32)):
            raise ValueError("ataOut_q must be [A, H1] and ataOut_s [A, H1/32]")
        if gmmY is None:
            gmmY = torch.empty(d.A, d.N1, dtype=torch.bfloat16, device=self.device)
        if d.want_permute_out:
            if permuteOut_q is None:
                permuteOut_q = torch.empty(d.A, d.H1, dtype=torch.uint8, device=self.device)
            if permuteOut_s is None:
                permuteOut_s = torch.empty(d.A, d.H1 // 32, dtype=torch.uint8, device=self.device)
        if d.BS:
            for t, name in ((mmX_q, "mmX_q"), (mmX_s, "mmX_s"), (mmWeight_q, "mmWeight_q"),
                            (mmWeight_s, "mmWeight_s")):
                _check(t, name, torch.uint8, 2)
            if mmY is None:
                mmY = torch.empty(d.BS, d.N2, dtype=torch.bfloat16, device=self.device)
        s = stream if stream is not None else torch.cuda.current_stream()
        args = (ctypes.byref(d), _ptr(ataOut_q) if d.A else None, _ptr(ataOut_s) if d.A else None,
                _ptr(recvCounts), _ptr(gmmWeight_q), _ptr(gmmWeight_s), _ptr(mmX_q) if d.BS else None,
                _ptr(mmX_s) if d.BS else None, _ptr(mmWeight_q) if d.BS else None,
                _ptr(mmWeight_s) if d.BS else None, _ptr(permuteOut_q) if d.want_permute_out else None,
                _ptr(permuteOut_s) if d.want_permute_out else None, _ptr(gmmY) if d.A else None,
                _ptr(mmY) if d.BS else None, _ptr(self.workspace), self.workspace.numel(),
                ctypes.c_void_p(s.cuda_stream))
        if gemm_events is None:
            name = "a2av_gmm_mx_run"
            st = load().a2av_gmm_mx_run(*args)
        else:
            name = "a2av_gmm_mx_run_profiled"
            for ev in gemm_events:
                if ev.cuda_event == 0:  # created lazily by torch: make it exist on this device
                    ev.record(s)
            st = load().a2av_gmm_mx_run_profiled(*args, ctypes.c_void_p(gemm_events[0].cuda_event),
                                                 ctypes.c_void_p(gemm_events[1].cuda_event))
        if st != A2AV_OK:
            raise A2avError(st, name)
        return gmmY, mmY, permuteOut_q, permuteOut_s
