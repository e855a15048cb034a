"""Dequantising rank reduce on the GPU against the float64 oracle (needs a GB300).

"aclnnQuantReduceScatter" page, Formula: out = sum over source ranks of
scales * data.  The kernel decodes exactly to float32, sums over ranks with
float32 fused multiply-adds (one rounding to nearest per rank), and rounds the
sum once to the output type.  With S = sum_w |value * scale| (float64), u32 =
2^-24 and u_out the output type's unit roundoff (2^-8 bf16, 2^-11 fp16, 2^-24
fp32), the error against the exact (float64) sum is at most

    u_out * |ref| + W * u32 * S * (1 + u_out) + (output subnormal step) + W * 2^-149

(W float32 roundings of partial sums, each at most u32 S; one final rounding:
u_out times the float32 sum; the last two terms cover underflow).  The bound
also holds for separately rounded products and sums, so it does not depend on
whether the kernel fuses them.
Every test uses this bound; NaN and infinity positions must match exactly.
"""

import numpy as np
import pytest
import torch

from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import (QREDUCE_WORKLOADS, QTYPE_NAMES, finite_codes,
                                                   quant_reduce_inputs)

pytestmark = pytest.mark.gpu

U_OUT = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11, torch.float32: 2.0 ** -24}  # 2^-(significant bits)
STEP_OUT = {torch.bfloat16: 2.0 ** -133, torch.float16: 2.0 ** -24, torch.float32: 2.0 ** -149}
QCODE = {"e4m3fn": 0, "e5m2": 1, "int8": 2}
MCODE = {"mx": 0, "group128": 1}
COMBOS = [("e4m3fn", "mx"), ("e5m2", "mx"), ("int8", "group128"), ("e4m3fn", "group128"),
          ("e5m2", "group128")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def gpu_reduce(data, scales, qtype, mode, out_dtype):
    dev = torch.device("cuda:0")
    W, rows, H = data.shape
    out = torch.empty(rows, H, dtype=out_dtype, device=dev)
    binding.a2av_quant_reduce(data.to(dev), scales.to(dev), qtype, mode, out)
    torch.cuda.synchronize()
    return out.cpu()


def abs_sum(orc, data, scales, qtype, mode):
    """S = sum over ranks of |value * scale| in float64, from the oracle's decoders."""
    W, rows, H = data.shape
    v = orc.decode8(QCODE[qtype], data.numpy())
    if mode == "mx":
        s = np.repeat(orc.decode8(3, scales.numpy()), 32, axis=2)
    else:
        s = np.repeat(scales.numpy().astype(np.float64), 128, axis=2)
    with np.errstate(invalid="ignore", over="ignore"):
        return np.abs(v * s).sum(0)


def assert_reduce_close(orc, got, data, scales, qtype, mode):
    ref = orc.quant_reduce(data.numpy(), scales.numpy(), QCODE[qtype], MCODE[mode])
    W = data.shape[0]
    g = got.double().numpy()
    nan_ref, nan_got = np.isnan(ref), np.isnan(g)
    assert np.array_equal(nan_ref, nan_got), np.argwhere(nan_ref != nan_got)[:5]
    inf_ref = np.isinf(ref)
    assert np.array_equal(np.isinf(g) & ~inf_ref, np.zeros_like(inf_ref)), np.argwhere(np.isinf(g) & ~inf_ref)[:5]
    assert np.array_equal(g[inf_ref], ref[inf_ref])
    fin = ~(nan_ref | inf_ref)
    S = abs_sum(orc, data, scales, qtype, mode)
    u = U_OUT[got.dtype]
    tol = u * np.abs(ref) + W * 2.0 ** -24 * S * (1 + u) + STEP_OUT[got.dtype] + W * 2.0 ** -149
    with np.errstate(invalid="ignore"):
        err = np.abs(g - ref)
    bad = fin & ~(err <= tol)
    assert not bad.any(), (np.argwhere(bad)[:5], g[bad][:5], ref[bad][:5], tol[bad][:5])


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("qtype,mode", COMBOS)
# Shapes: below one 256-unit chunk (direct loads only); scale planes that do
# not start on 16 bytes (direct loads only); whole chunks staged through shared
# memory; staged chunks plus a direct-load tail.
@pytest.mark.parametrize("W,rows,H", [(2, 1, 1024), (4, 37, 1152), (8, 5, 8192), (2, 45, 1024)])
def test_matches_oracle(orc, qtype, mode, out_dtype, W, rows, H):
    # fp16 output: keep |sum| <= 8 * 57344 * 2^-4 < 65504, so no output overflows.
    er = (-12, -4) if out_dtype == torch.float16 else (-10, 6)
    data, scales = quant_reduce_inputs(W, rows, H, qtype, mode, seed=W * 1000 + rows, exp_range=er)
    got = gpu_reduce(data, scales, qtype, mode, out_dtype)
    assert_reduce_close(orc, got, data, scales, qtype, mode)


@pytest.mark.parametrize("qtype", QTYPE_NAMES)
def test_every_code_once(orc, qtype):
    # Each finite code of the format at unit scale, one per element: exact decode.
    codes = finite_codes(qtype)
    H = 1024
    row = np.resize(codes, H).astype(np.uint8)
    data = torch.from_numpy(np.stack([row[None, :], np.zeros((1, H), np.uint8)]))  # W = 2, rows = 1
    mode = "group128" if qtype == "int8" else "mx"
    if mode == "mx":
        scales = torch.full((2, 1, H // 32), 127, dtype=torch.uint8)
    else:
        scales = torch.ones(2, 1, H // 128, dtype=torch.float32)
    got = gpu_reduce(data, scales, qtype, mode, torch.float32)
    assert np.array_equal(got.double().numpy()[0], orc.decode8(QCODE[qtype], row))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_nan_inf_and_subnormal_codes(orc, out_dtype):
    W, rows, H = 2, 6, 1024
    for qtype in ("e4m3fn", "e5m2"):
        data, scales = quant_reduce_inputs(W, rows, H, qtype, "mx", seed=5, exp_range=(-12, -4))
        d, s = data.numpy().copy(), scales.numpy().copy()
        if qtype == "e4m3fn":
            d[0, 0, 5] = 0x7F                    # NaN
            d[1, 2, 100] = 0xFF                  # NaN, negative sign bit
            d[:, 5, 0:32] = 0x01                 # smallest subnormal, 2^-9 ...
            s[:, 5, 0] = 0                       # ... times 2^-127: a float32 subnormal product
        else:
            d[0, 1, 7], d[1, 1, 7] = 0x7C, 0xFC  # +inf + -inf = NaN
            d[0, 3, 9] = 0x7C                    # +inf alone
            d[1, 3, 10] = 0xFC                   # -inf alone
            d[0, 2, 11] = 0x7D                   # NaN
            d[:, 5, 0:32] = 0x01                 # 2^-16 times 2^-127
            s[:, 5, 0] = 0
        s[1, 4, 3] = 0xFF                        # E8M0 NaN scale: the whole 32-element group
        data, scales = torch.from_numpy(d), torch.from_numpy(s)
        got = gpu_reduce(data, scales, qtype, "mx", out_dtype)
        assert_reduce_close(orc, got, data, scales, qtype, "mx")
        assert torch.isnan(got[4, 96:128].float()).all()


def test_output_overflow(orc):
    W, rows, H = 8, 2, 1024
    data = torch.full((W, rows, H), 0x7E, dtype=torch.uint8)     # E4M3 448
    scales = torch.full((W, rows, H // 32), 127 + 7, dtype=torch.uint8)
    # 8 * 448 * 2^7 = 458752: finite in bf16 and float32, beyond fp16's 65504.
    got16 = gpu_reduce(data, scales, "e4m3fn", "mx", torch.float16)
    assert torch.isinf(got16.float()).all() and (got16.float() > 0).all()
    for dt in (torch.bfloat16, torch.float32):
        assert_reduce_close(orc, gpu_reduce(data, scales, "e4m3fn", "mx", dt), data, scales, "e4m3fn", "mx")


def test_unaligned_scales_take_the_direct_path(orc):
    # Float scales 4-byte but not 16-byte aligned: the bulk copies need 16, so
    # every unit is loaded directly; the results must not change.
    data, scales = quant_reduce_inputs(4, 64, 2048, "int8", "group128", seed=6)
    dev = torch.device("cuda:0")
    flat = torch.empty(scales.numel() + 1, dtype=torch.float32, device=dev)
    odd = flat[1:].view(scales.shape)
    odd.copy_(scales.to(dev))
    assert odd.data_ptr() % 16 != 0
    out = torch.empty(64, 2048, dtype=torch.bfloat16, device=dev)
    binding.a2av_quant_reduce(data.to(dev), odd, "int8", "group128", out)
    aligned = gpu_reduce(data, scales, "int8", "group128", torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), aligned.view(torch.int16))
    assert_reduce_close(orc, aligned, data, scales, "int8", "group128")


def test_side_stream_and_determinism(orc):
    data, scales = quant_reduce_inputs(4, 300, 2048, "int8", "group128", seed=3)
    dev = torch.device("cuda:0")
    d, s = data.to(dev), scales.to(dev)
    side = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        o = torch.full((300, 2048), float("nan"), dtype=torch.bfloat16, device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            binding.a2av_quant_reduce(d, s, "int8", "group128", o, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        outs.append(o.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_reduce_close(orc, outs[0], data, scales, "int8", "group128")


@pytest.mark.parametrize("name", list(QREDUCE_WORKLOADS))
def test_full_size_workload(orc, name):
    # The configuration the benchmark times, compared on sampled rows (rows reduce independently).
    wl = QREDUCE_WORKLOADS[name]
    data, scales = quant_reduce_inputs(wl.W, wl.rows, wl.H, wl.qtype, wl.mode, seed=0)
    got = gpu_reduce(data, scales, wl.qtype, wl.mode, torch.bfloat16)
    rng = np.random.default_rng(11)
    idx = np.unique(np.concatenate([[0, wl.rows - 1], rng.integers(0, wl.rows, 24)]))
    assert_reduce_close(orc, got[idx], data[:, idx].contiguous(), scales[:, idx].contiguous(), wl.qtype, wl.mode)
