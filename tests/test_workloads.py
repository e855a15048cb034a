"""Seeded input generator self-checks (CPU only)."""

import numpy as np
import torch

from token_permute_grouped_gb300 import workloads as wk


def test_counts_deterministic_and_summing():
    for name in ("tiny_w2e2_h256_n128", "w8e4_h4096_n1024_shared2048", "skew_w8e32_h4096_n1536_fp16"):
        wl = wk.WORKLOADS[name]
        a = wk.recv_counts(wl, 0)
        b = wk.recv_counts(wl, 0)
        assert a.dtype == np.int32 and a.shape == (wl.W * wl.e,)
        assert np.array_equal(a, b) and (a >= 0).all()
    assert wk.recv_counts(wk.WORKLOADS["tiny_w2e2_h256_n128"]).sum() == 256


def test_skew_forced_empties():
    wl = wk.WORKLOADS["skew_w8e32_h4096_n1536_fp16"]
    rc = wk.recv_counts(wl, 0)
    assert (rc == 0).sum() == round(0.2 * wl.W * wl.e)
    groups = rc.reshape(wl.W, wl.e).sum(0)
    assert (groups == 0).sum() == (round(0.2 * wl.W * wl.e)) // wl.W


def test_tensor_values_independent_of_thread_count(monkeypatch):
    n = 3 * (1 << 22) + 5
    a = wk.normal_f32(n, 0, 1)
    monkeypatch.setattr(wk.os, "cpu_count", lambda: 1)
    b = wk.normal_f32(n, 0, 1)
    assert np.array_equal(a, b)


def test_tiny_inputs_shapes():
    inp = wk.make_inputs(wk.WORKLOADS["tiny_w2e2_h256_n128"])
    assert inp.ataOut.shape == (256, 256) and inp.ataOut.dtype == torch.bfloat16
    assert inp.gmmWeight.shape == (2, 256, 128)
    assert inp.mmX is None
    # ataOut ~ N(0,1)/sqrt(H1) for this workload
    assert abs(inp.ataOut.float().std().item() - 1 / 16) < 0.01


def test_random_counts_sum_and_zeros():
    for A in (0, 1, 77):
        rc = wk.random_counts(4, 3, A, seed=1, zero_prob=0.5)
        assert rc.sum() == A and (rc >= 0).all()
