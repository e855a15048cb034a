"""The oracle's results do not depend on its thread count: every output row
is one sequential float64 sum over k, whichever thread computes it (the
CPU baseline times it on one core and on all of them)."""

import numpy as np
import torch

from token_permute_grouped_gb300.workloads import custom_inputs, random_counts


def test_grouped_product_same_bits_on_one_and_many_threads(orc):
    inp = custom_inputs(4, 3, 256, 96, random_counts(4, 3, 700, 5, 0.2), "bf16", 90, 128, 40, seed=5)
    wl = inp.wl
    n = orc.num_threads()
    try:
        orc.set_threads(1)
        one = orc.run(wl.W, wl.e, inp.recvCounts, inp.ataOut, inp.gmmWeight, inp.mmX, inp.mmWeight)
        orc.set_threads(max(2, n))
        many = orc.run(wl.W, wl.e, inp.recvCounts, inp.ataOut, inp.gmmWeight, inp.mmX, inp.mmWeight)
    finally:
        orc.set_threads(n)
    assert torch.equal(one[0].view(torch.int16), many[0].view(torch.int16))  # permuteOut
    assert np.array_equal(one[1], many[1]) and np.array_equal(one[2], many[2])
