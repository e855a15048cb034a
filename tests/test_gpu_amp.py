"""Dynamic loss scaling on the GPU against the oracle (needs a GB300).

The scale update follows the "aclnnAmpUpdateScale" page's formula in float32,
so the GPU must match the oracle bit for bit, including the overflow and
NaN cases.  The inf/NaN scan must find any planted non-finite value, in the
16-byte vector body and in the tail, and otherwise leave the flag alone.
"""

import numpy as np
import pytest
import torch

from token_permute_grouped_gb300 import binding, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        iv = int(rng.choice([1, 2, 3, 7, 2000, 2**31 - 1]))
        tr = int(rng.integers(0, min(iv, 5)))
        if rng.random() < 0.3:
            tr = iv - 1  # growth step
        sc = float(np.float32(rng.choice([1.0, 65536.0, 3.0e38, 1.0e-38, float(2.0 ** rng.integers(-30, 30))])))
        fi = float(rng.choice([0.0, 0.0, 0.0, 1.0, -2.0, float("inf"), float("nan")]))
        gr = float(rng.choice([2.0, 1.5, 1.0e30]))
        bo = float(rng.choice([0.5, 0.25, 1.0e-30]))
        yield sc, tr, fi, gr, bo, iv


def test_update_matches_oracle_bitwise(orc):
    dev = torch.device("cuda:0")
    for sc, tr, fi, gr, bo, iv in _cases(300, 1):
        s = torch.tensor([sc], dtype=torch.float32, device=dev)
        t = torch.tensor([tr], dtype=torch.int32, device=dev)
        f = torch.tensor([fi], dtype=torch.float32, device=dev)
        binding.a2av_amp_update_scale(s, t, f, gr, bo, iv)
        want_s, want_t = orc.amp_update_scale(sc, tr, fi, gr, bo, iv)
        assert int(t.item()) == want_t, (sc, tr, fi, gr, bo, iv)
        assert s.cpu().numpy().tobytes() == np.float32(want_s).tobytes(), (sc, tr, fi, gr, bo, iv, s.item(), want_s)


def test_update_sequence_matches_oracle(orc):
    # A training-loop-like sequence: the state carries over between calls.
    dev = torch.device("cuda:0")
    s = torch.tensor([65536.0], dtype=torch.float32, device=dev)
    t = torch.zeros(1, dtype=torch.int32, device=dev)
    ref_s, ref_t = 65536.0, 0
    rng = np.random.default_rng(2)
    for _ in range(200):
        fi = 1.0 if rng.random() < 0.05 else 0.0
        binding.a2av_amp_update_scale(s, t, torch.tensor([fi], device=dev), 2.0, 0.5, 7)
        ref_s, ref_t = orc.amp_update_scale(ref_s, ref_t, fi, 2.0, 0.5, 7)
    assert s.item() == ref_s and int(t.item()) == ref_t


def test_update_rejects_bad_interval():
    dev = torch.device("cuda:0")
    s = torch.ones(1, device=dev)
    t = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(binding.A2avError):
        binding.a2av_amp_update_scale(s, t, torch.zeros(1, device=dev), 2.0, 0.5, 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 4099, 1 << 20])
def test_nonfinite_scan(orc, dtype, n):
    dev = torch.device("cuda:0")
    gen = torch.Generator().manual_seed(n)
    x = torch.randn(n, generator=gen).to(dtype)
    flag = torch.zeros(1, dtype=torch.float32, device=dev)
    binding.a2av_found_nonfinite(x.to(dev), flag)
    assert flag.item() == 0.0 and not orc.any_nonfinite(x)
    # The flag is only ever raised: a finite tensor leaves a set flag set.
    flag.fill_(1.0)
    binding.a2av_found_nonfinite(x.to(dev), flag)
    assert flag.item() == 1.0
    for pos in sorted({0, n - 1, n // 2, max(0, n - 3)}):
        for bad in (float("inf"), float("-inf"), float("nan")):
            y = x.clone()
            y[pos] = bad
            flag.zero_()
            binding.a2av_found_nonfinite(y.to(dev), flag)
            assert flag.item() == 1.0 and orc.any_nonfinite(y), (pos, bad)


def test_scan_and_update_after_the_hot_path(orc):
    # The loss-scale step as a training loop would run it on the layer output.
    from gpu_helpers import run_gpu
    from token_permute_grouped_gb300.workloads import custom_inputs
    inp = custom_inputs(2, 2, 128, 64, [40, 2, 0, 90], "fp16", 0, 0, 0, seed=9)
    gmmY, _, _, (st, _) = run_gpu(inp, "default", want_perm=False)
    assert st == 0
    dev = torch.device("cuda:0")
    for plant in (False, True):
        y = gmmY.clone()
        if plant:
            y[3, 5] = float("inf")
        flag = torch.zeros(1, device=dev)
        binding.a2av_found_nonfinite(y.to(dev), flag)
        s = torch.tensor([1024.0], device=dev)
        t = torch.tensor([4], dtype=torch.int32, device=dev)
        binding.a2av_amp_update_scale(s, t, flag, 2.0, 0.5, 100)
        want = orc.amp_update_scale(1024.0, 4, 1.0 if orc.any_nonfinite(y) else 0.0, 2.0, 0.5, 100)
        assert (s.item(), int(t.item())) == want
