"""Arrival-driven start (a2av_gmm_run_arrivals) on one GPU.

"aclnnAlltoAllvGroupedMatMul", API function and Formula: ataOut =
AlltoAllv(gmmX), then Permute and GroupedMatMul.  Here the kernel is launched
before the rows are there: a second stream plays the exchange, copying each
source's rows into ataOut (from pinned host memory, on a copy engine) and
then that source's flag.  The kernel runs the shared expert first and makes
each routed tile wait for the flags of the sources its rows come from.

- ataOut starts out holding NaN: a tile that read a row before its source
  arrived would give NaN or wrong products, and the oracle check would fail;
- the copies are enqueued only after the kernel has been running for a few
  milliseconds, so the waits are really exercised;
- a source whose flag is never set makes the kernel give up after the wait
  limit (20 ms here) and report A2AV_ERR_ARRIVAL_TIMEOUT, and the next call
  on the same device works.
"""

import time

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, check_full
from token_permute_grouped_gb300 import binding, build
from token_permute_grouped_gb300.workloads import custom_inputs, random_counts

pytestmark = pytest.mark.gpu

NAN_BITS = 0x7FC1  # bf16 and fp16 NaN


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def _case(dtype="bf16", want_shared=True, seed=31):
    W, e = 8, 4
    rc = random_counts(W, e, 6000, seed, 0.1)
    if want_shared:
        return custom_inputs(W, e, 512, 256, rc, dtype, 2048, 512, 512, seed=seed)
    return custom_inputs(W, e, 512, 256, rc, dtype, seed=seed)


def _source_spans(inp):
    """Rows [begin, end) of ataOut that each source rank sends (its e runs, rank-major)."""
    W, e = inp.wl.W, inp.wl.e
    per_source = inp.recvCounts.reshape(W, e).astype(np.int64).sum(1)
    ends = np.cumsum(per_source)
    return [(int(b), int(t)) for b, t in zip(ends - per_source, ends)]


def _setup(inp, want_perm, tiles="default"):
    wl = inp.wl
    dev = torch.device("cuda:0")
    dt = wl.torch_dtype
    d = binding.make_desc(wl.W, wl.e, inp.A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, dt,
                          want_permute_out=want_perm, path="fused", tiles=tiles)
    t = dict(
        ata=torch.empty(inp.A, wl.H1, dtype=dt, device=dev),
        rc=torch.from_numpy(inp.recvCounts).to(dev),
        gw=inp.gmmWeight.to(dev),
        mmX=inp.mmX.to(dev) if wl.BS else None,
        mmW=inp.mmWeight.to(dev) if wl.BS else None,
        y=torch.empty(inp.A, wl.N1, dtype=dt, device=dev),
        mmY=torch.empty(wl.BS, wl.N2, dtype=dt, device=dev) if wl.BS else None,
        perm=torch.empty(inp.A, wl.H1, dtype=dt, device=dev) if want_perm else None,
        ws=torch.empty(binding.a2av_gmm_workspace_size(d), dtype=torch.uint8, device=dev),
        arrived=torch.zeros(wl.W, dtype=torch.int64, device=dev),
    )
    t["ata"].view(torch.int16).fill_(NAN_BITS)
    return d, t


def _launch(d, t, tag, limit_ns):
    binding.a2av_gmm_run_arrivals(d, t["ata"], t["rc"], t["gw"], t["mmX"], t["mmW"], t["perm"], t["y"], t["mmY"],
                                  t["arrived"], tag, limit_ns, t["ws"])


def _exchange_buffers(inp, tag):
    """Pinned host copies and the side stream, made before any kernel is
    launched: a pinned allocation may wait for the device, and the kernel
    waits for these very copies."""
    return torch.cuda.Stream(), inp.ataOut.pin_memory(), torch.tensor([tag], dtype=torch.int64).pin_memory()


def _exchange(inp, t, bufs, order, skip=None):
    """On a side stream: each source's rows, then its flag, in `order` (copies only)."""
    side, host_rows, host_tag = bufs
    spans = _source_spans(inp)
    with torch.cuda.stream(side):
        for w in order:
            b, e = spans[w]
            if e > b:
                t["ata"][b:e].copy_(host_rows[b:e], non_blocking=True)
            if w != skip:
                t["arrived"][w:w + 1].copy_(host_tag, non_blocking=True)
    return side


# The kernel takes the routed row tiles in the order of the latest source
# their rows come from (up to 2048 row tiles; beyond that, group order):
# both orders, single-CTA and pair tiles.
CASES = {
    "bf16": lambda: _case("bf16"),
    "fp16": lambda: _case("fp16"),
    # 32 experts of about 8,800 rows: 128-row tiles on one CTA give more than
    # 2048 row tiles (group order), 256-row pair tiles fewer (arrival order).
    "over_order_capacity": lambda: custom_inputs(4, 32, 128, 128, [2000 + (i * 37) % 400 for i in range(128)],
                                                 "bf16", 256, 128, 128, seed=34),
    # 32 sources, a quarter of them sending nothing (their flags still
    # arrive), runs of 0 to 300 rows.
    "many_sources_some_empty": lambda: custom_inputs(
        32, 2, 256, 192, [0 if (i // 2) % 4 == 3 else (i * 53) % 301 for i in range(64)], "fp16", 100, 128, 64,
        seed=35),
}


def test_order_capacity_case_spans_both_orders():
    rc = np.array([2000 + (i * 37) % 400 for i in range(128)]).reshape(4, 32).sum(0)
    assert sum(-(-int(g) // 128) for g in rc) > 2048
    assert sum(-(-int(g) // 256) for g in rc) <= 2048


@pytest.mark.parametrize("want_perm", [False, True])
@pytest.mark.parametrize("tiles", ["pair", "single"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_rows_arriving_during_the_kernel(orc, case, tiles, want_perm):
    inp = CASES[case]()
    d, t = _setup(inp, want_perm, tiles)
    tag = int(np.random.default_rng(7).integers(1, 2**62))
    bufs = _exchange_buffers(inp, tag)
    torch.cuda.synchronize()
    _launch(d, t, tag, 2_000_000_000)
    time.sleep(0.005)  # the kernel is running and its routed tiles are waiting
    order = np.random.default_rng(8).permutation(inp.wl.W).tolist()
    _exchange(inp, t, bufs, order)
    torch.cuda.synchronize()
    st, code = binding.a2av_gmm_read_device_status(t["ws"])
    assert (st, code) == (0, 0), (st, code)
    y, m = t["y"].cpu(), t["mmY"].cpu() if t["mmY"] is not None else None
    perm = t["perm"].cpu() if want_perm else None
    check_full(orc, inp, y, m, perm)
    # The same bits as the ordinary call of the fused path on the arrived rows.
    plan = binding.Plan(inp.wl.W, inp.wl.e, inp.A, inp.wl.H1, inp.wl.N1, inp.wl.BS, inp.wl.H2, inp.wl.N2,
                        inp.wl.torch_dtype, path="fused", tiles=tiles)
    y2, m2, _ = plan.run(t["ata"], t["rc"], t["gw"], t["mmX"], t["mmW"])
    torch.cuda.synchronize()
    assert_bits_equal(y, y2.cpu(), "gmmY")
    if m is not None:
        assert_bits_equal(m, m2.cpu(), "mmY")


def test_everything_arrived_before_the_launch(orc):
    inp = _case("bf16", want_shared=False, seed=32)
    d, t = _setup(inp, False)
    tag = 12345
    side = _exchange(inp, t, _exchange_buffers(inp, tag), list(range(inp.wl.W)))
    side.synchronize()
    _launch(d, t, tag, 0)
    torch.cuda.synchronize()
    assert binding.a2av_gmm_read_device_status(t["ws"]) == (0, 0)
    check_full(orc, inp, t["y"].cpu(), None, None)


def test_a_source_that_never_arrives_times_out():
    inp = _case("bf16", seed=33)
    d, t = _setup(inp, False)
    tag = 777
    missing = int(np.argmax(inp.recvCounts.reshape(inp.wl.W, inp.wl.e).sum(1)))
    side = _exchange(inp, t, _exchange_buffers(inp, tag), list(range(inp.wl.W)), skip=missing)
    side.synchronize()
    t0 = time.perf_counter()
    _launch(d, t, tag, 20_000_000)  # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    st, code = binding.a2av_gmm_read_device_status(t["ws"])
    assert binding.STATUS_NAMES[st] == "A2AV_ERR_ARRIVAL_TIMEOUT" and code & 8, (st, code)
    assert elapsed < 10.0
    # The device is fine afterwards: the flag arrives and a new call succeeds.
    t["arrived"][missing] = tag
    _launch(d, t, tag, 0)
    torch.cuda.synchronize()
    assert binding.a2av_gmm_read_device_status(t["ws"]) == (0, 0)
