"""Pins for the CPU oracle: facts fixed by the operator page or by mathematics.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with something other than itself: hand-worked fixtures, the sum
rule and bijection of Permute, cases that reduce to a library routine (numpy
float64 matmul, numpy/torch float decoding), exact identity / one-hot /
integer cases, and brute force on tiny inputs.  The same pins run against
deliberately broken builds of the oracle (test_oracle_mutants.py) to show
that each plausible mistake is caught.

Pages cited: "aclnnAlltoAllvGroupedMatMul", sections "Formula"
(permuteOut = Permute(ataOut), gmmY = permuteOut x gmmWeight,
mmY = mmX x mmWeight) and "Shape variables" (A = sum of recvCounts);
"aclnnAmpUpdateScale", "Formula" and its notes, for the loss-scale update;
"aclnnQuantReduceScatter", "Formula" and "Constraints" (mx quantisation:
FLOAT8 codes with one FLOAT8_E8M0 scale per 32 elements; float scales per
128), for the quantised reduce and the block-scaled FP8 grouped product.
"""

from __future__ import annotations

import json
import os

import numpy as np
import torch

from oracle import OracleError
from token_permute_grouped_gb300.workloads import random_counts

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _expert_of_arrival_rows(W, e, rc):
    """Brute force: the local expert of every ataOut row, in arrival order."""
    out = []
    for w in range(W):
        for j in range(e):
            out += [j] * int(rc[w * e + j])
    return out


def _tagged(A, H, dtype):
    """Row r carries r in base-256 digits in columns 0..2 (exact in bf16/fp16)."""
    t = torch.zeros(A, H, dtype=torch.float64)
    r = torch.arange(A, dtype=torch.float64)
    t[:, 0] = torch.floor(r / 65536)
    t[:, 1] = torch.floor(r / 256) % 256
    t[:, 2] = r % 256
    if H > 3:
        t[:, 3:] = torch.randn(A, H - 3, generator=torch.Generator().manual_seed(A), dtype=torch.float64)
    return t.to(dtype)


def _untag(t):
    v = t[:, :3].to(torch.float64)
    return (v[:, 0] * 65536 + v[:, 1] * 256 + v[:, 2]).to(torch.int64)


def _small_cases():
    # (W, e, A, zero_prob, seed): several shapes, with empty segments/groups.
    return [(1, 1, 5, 0.0, 0), (1, 4, 9, 0.3, 1), (3, 1, 8, 0.0, 2), (2, 2, 6, 0.5, 3),
            (4, 3, 40, 0.4, 4), (8, 4, 100, 0.25, 5), (2, 8, 0, 0.0, 6), (5, 2, 1, 0.0, 7)]


# ---- decoding ----------------------------------------------------------------

def pin_decode_bf16_all_patterns(orc):
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.bfloat16)
    got = orc.decode(t)
    want = t.to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_decode_fp16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.float16)
    got = orc.decode(t)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# ---- plan / permute -------------------------------------------------------------

def pin_plan_golden(orc):
    g = _golden("permute_w2e3.json")
    src, dst, gr, go = orc.plan(g["W"], g["e"], g["recvCounts"], g["A"])
    assert src.tolist() == g["src_off"]
    assert dst.tolist() == g["dst_off"]
    assert gr.tolist() == g["group_rows"]
    assert go.tolist() == g["group_off"]


def pin_plan_rejects_bad_counts(orc):
    # Sum rule: A is the sum of recvCounts; negative counts are meaningless.
    for rc, A in [([1, 2, 3, 4], 9), ([1, 2, 3, 4], 11), ([1, -1, 3, 4], 7)]:
        try:
            orc.plan(2, 2, rc, A)
        except OracleError:
            continue
        raise AssertionError(f"plan accepted recvCounts={rc} with A={A}")


def pin_permute_golden(orc):
    g = _golden("permute_w2e3.json")
    ata = _tagged(g["A"], 8, torch.bfloat16)
    perm = orc.permute(g["W"], g["e"], g["recvCounts"], ata)
    assert _untag(perm).tolist() == g["permuted_source_rows"]
    assert torch.equal(perm.view(torch.int16), ata[g["permuted_source_rows"]].view(torch.int16))


def pin_permute_matches_stable_sort(orc):
    # Brute force: Permute is a stable sort of the arrival rows by local expert.
    for W, e, A, zp, seed in _small_cases():
        rc = random_counts(W, e, A, seed, zp)
        experts = _expert_of_arrival_rows(W, e, rc)
        want = sorted(range(A), key=lambda r: experts[r])
        ata = _tagged(A, 4, torch.bfloat16)
        perm = orc.permute(W, e, rc, ata)
        assert _untag(perm).tolist() == want, (W, e, rc.tolist())


def pin_permute_is_bijection_preserving_rows(orc):
    for W, e, A, zp, seed in _small_cases() + [(16, 16, 3000, 0.1, 11)]:
        rc = random_counts(W, e, A, seed, zp)
        ata = _tagged(A, 16, torch.float16)
        perm = orc.permute(W, e, rc, ata)
        idx = _untag(perm)
        assert sorted(idx.tolist()) == list(range(A))
        assert torch.equal(perm.view(torch.int16), ata[idx].view(torch.int16))


def pin_permute_identity_cases(orc):
    # W = 1 or e = 1: arrival order already is expert order.
    for W, e, A, seed in [(1, 1, 17, 0), (1, 6, 50, 1), (7, 1, 33, 2)]:
        rc = random_counts(W, e, A, seed, 0.2)
        ata = torch.randn(A, 24, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        perm = orc.permute(W, e, rc, ata)
        assert torch.equal(perm.view(torch.int16), ata.view(torch.int16))


def pin_group_rows_sum_rule(orc):
    for W, e, A, zp, seed in _small_cases():
        rc = random_counts(W, e, A, seed, zp)
        _, _, gr, go = orc.plan(W, e, rc, A)
        assert gr.tolist() == rc.reshape(W, e).sum(0).tolist()
        assert go[-1] == A and go[0] == 0


# ---- grouped matmul -------------------------------------------------------------

def _to16(x, dtype):
    return torch.tensor(np.asarray(x, dtype=np.float64)).to(dtype)


def pin_grouped_matmul_golden(orc):
    g = _golden("grouped_matmul_w2e2.json")
    for dtype in (torch.bfloat16, torch.float16):
        ata = _to16(g["ataOut"], dtype)
        w = _to16(g["gmmWeight"], dtype)
        perm, y, _ = orc.run(g["W"], g["e"], g["recvCounts"], ata, w)
        assert perm.to(torch.float64).tolist() == g["permuteOut"]
        assert y.tolist() == g["gmmY"]
        mm = orc.matmul(_to16(g["mmX"], dtype), _to16(g["mmWeight"], dtype))
        assert mm.tolist() == g["mmY"]


def pin_single_group_is_numpy_matmul(orc):
    # W = 1, e = 1: one plain product; numpy's float64 matmul is the library check.
    rng = np.random.default_rng(5)
    for A, H, N, dtype in [(33, 40, 24, torch.bfloat16), (64, 128, 72, torch.float16), (1, 8, 8, torch.bfloat16)]:
        x = torch.from_numpy(rng.standard_normal((A, H))).to(dtype)
        w = torch.from_numpy(rng.standard_normal((1, H, N))).to(dtype)
        _, y, _ = orc.run(1, 1, [A], x, w)
        ref = x.to(torch.float64).numpy() @ w[0].to(torch.float64).numpy()
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def pin_grouped_blocks_match_numpy(orc):
    # Each expert block of gmmY is a standalone product of that block.
    rng = np.random.default_rng(6)
    for W, e, A, zp, seed in [(2, 2, 50, 0.0, 1), (4, 3, 70, 0.4, 2), (3, 5, 0, 0.0, 3)]:
        rc = random_counts(W, e, A, seed, zp)
        H, N = 48, 40
        x = torch.from_numpy(rng.standard_normal((A, H))).to(torch.bfloat16)
        w = torch.from_numpy(rng.standard_normal((e, H, N))).to(torch.bfloat16)
        perm, y, _ = orc.run(W, e, rc, x, w)
        experts = _expert_of_arrival_rows(W, e, rc)
        order = sorted(range(A), key=lambda r: experts[r])
        xs = x.to(torch.float64).numpy()
        start = 0
        for j in range(e):
            rows = [r for r in order if experts[r] == j]
            if rows:
                ref = xs[rows] @ w[j].to(torch.float64).numpy()
                np.testing.assert_allclose(y[start:start + len(rows)], ref, rtol=1e-12, atol=1e-12)
            start += len(rows)
        assert start == A


def pin_identity_weight_exact(orc):
    # gmmWeight[j] = I  =>  gmmY == permuteOut exactly.
    W, e, A, H = 3, 4, 90, 32
    rc = random_counts(W, e, A, 9, 0.3)
    x = torch.randn(A, H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    w = torch.eye(H).repeat(e, 1, 1).to(torch.bfloat16)
    perm, y, _ = orc.run(W, e, rc, x, w)
    assert np.array_equal(y, perm.to(torch.float64).numpy())


def pin_scaled_one_hot_weight_exact(orc):
    # gmmWeight[j][k][n] = 2^j [k == pi(n)]  =>  gmmY[i][n] = 2^{j(i)} permuteOut[i][pi(n)].
    W, e, A, H, N = 2, 5, 80, 24, 16
    rc = random_counts(W, e, A, 4, 0.3)
    pi = np.random.default_rng(3).permutation(H)[:N]
    w = torch.zeros(e, H, N, dtype=torch.float64)
    for j in range(e):
        w[j, pi, np.arange(N)] = 2.0 ** j
    x = torch.randn(A, H, generator=torch.Generator().manual_seed(2)).to(torch.float16)
    perm, y, _ = orc.run(W, e, rc, x, w.to(torch.float16))
    _, _, gr, _ = orc.plan(W, e, rc, A)
    scale = np.repeat(2.0 ** np.arange(e), gr)
    want = perm.to(torch.float64).numpy()[:, pi] * scale[:, None]
    assert np.array_equal(y, want)


def pin_one_hot_activations_exact(orc):
    # Arrival row r = unit vector e_{k(r)}  =>  its gmmY row = gmmWeight[j(r)][k(r)].
    W, e, A, H, N = 3, 3, 45, 20, 12
    rc = random_counts(W, e, A, 8, 0.2)
    k_of = np.random.default_rng(4).integers(0, H, A)
    x = torch.zeros(A, H, dtype=torch.float64)
    x[np.arange(A), k_of] = 1.0
    w = torch.randn(e, H, N, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    _, y, _ = orc.run(W, e, rc, x.to(torch.bfloat16), w)
    experts = _expert_of_arrival_rows(W, e, rc)
    order = sorted(range(A), key=lambda r: experts[r])
    wd = w.to(torch.float64).numpy()
    want = np.stack([wd[experts[r], k_of[r]] for r in order])
    assert np.array_equal(y, want)


def pin_integer_inputs_exact(orc):
    # Small integers: every partial sum is an integer far below 2^53, so the
    # result is exact and equals numpy's int64 product.
    rng = np.random.default_rng(7)
    W, e, A, H, N = 4, 2, 60, 64, 24
    rc = random_counts(W, e, A, 10, 0.2)
    xi = rng.integers(-4, 5, (A, H))
    wi = rng.integers(-4, 5, (e, H, N))
    x = torch.tensor(xi, dtype=torch.float64).to(torch.bfloat16)
    w = torch.tensor(wi, dtype=torch.float64).to(torch.bfloat16)
    _, y, _ = orc.run(W, e, rc, x, w)
    experts = _expert_of_arrival_rows(W, e, rc)
    order = sorted(range(A), key=lambda r: experts[r])
    want = np.stack([xi[r] @ wi[experts[r]] for r in order]) if A else np.zeros((0, N))
    assert np.array_equal(y, want.astype(np.float64))


def pin_row_subset_equals_full(orc):
    W, e, A, H, N = 2, 3, 40, 16, 8
    rc = random_counts(W, e, A, 12, 0.2)
    x = torch.randn(A, H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    w = torch.randn(e, H, N, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    perm, full, _ = orc.run(W, e, rc, x, w)
    _, _, gr, _ = orc.plan(W, e, rc, A)
    rows = [A - 1, 0, 7, 7, 19]
    sub = orc.grouped_matmul(gr, perm, w, rows)
    assert np.array_equal(sub, full[rows])


# ---- shared expert ---------------------------------------------------------------

def pin_shared_matmul_numpy(orc):
    rng = np.random.default_rng(8)
    for BS, H, N, dtype in [(17, 40, 24, torch.bfloat16), (32, 64, 48, torch.float16)]:
        x = torch.from_numpy(rng.standard_normal((BS, H))).to(dtype)
        w = torch.from_numpy(rng.standard_normal((H, N))).to(dtype)
        y = orc.matmul(x, w)
        ref = x.to(torch.float64).numpy() @ w.to(torch.float64).numpy()
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
        rows = [BS - 1, 3]
        assert np.array_equal(orc.matmul(x, w, rows), y[rows])


def pin_shared_identity_and_integer_exact(orc):
    rng = np.random.default_rng(9)
    x = torch.randn(12, 16, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    y = orc.matmul(x, torch.eye(16).to(torch.bfloat16))
    assert np.array_equal(y, x.to(torch.float64).numpy())
    xi = rng.integers(-4, 5, (20, 96))
    wi = rng.integers(-4, 5, (96, 40))
    y = orc.matmul(torch.tensor(xi, dtype=torch.float64).to(torch.float16),
                   torch.tensor(wi, dtype=torch.float64).to(torch.float16))
    assert np.array_equal(y, (xi @ wi).astype(np.float64))


# ---- AMP loss-scale update (page "aclnnAmpUpdateScale") ---------------------

def pin_amp_update_golden(orc):
    g = _golden("amp_update_scale.json")
    for sc, tr, fi, gr, bo, iv, want_sc, want_tr in g["cases"]:
        got_sc, got_tr = orc.amp_update_scale(sc, tr, fi, gr, bo, iv)
        assert got_tr == want_tr, (sc, tr, fi, iv, got_tr)
        assert np.float32(got_sc) == np.float32(want_sc), (sc, tr, fi, iv, got_sc)
    c = g["nan_found_inf_case"]
    got = orc.amp_update_scale(c["scale"], c["tracker"], float("nan"), c["growth"], c["backoff"], c["interval"])
    assert got == (c["want_scale"], c["want_tracker"])


def pin_amp_update_rejects_bad_interval(orc):
    for iv in (0, -5):
        try:
            orc.amp_update_scale(1.0, 0, 0.0, 2.0, 0.5, iv)
        except OracleError:
            continue
        raise AssertionError(f"growth_interval {iv} accepted")


def pin_amp_update_matches_torch(orc):
    # torch's own CPU routine for the same update, as a library check.
    rng = np.random.default_rng(11)
    for _ in range(400):
        iv = int(rng.integers(1, 6))
        tr = int(rng.integers(0, iv))
        sc = float(np.float32(rng.choice([1.0, 65536.0, 3.0e38, 1e-30, 2.0 ** rng.integers(-20, 20)])))
        fi = float(rng.choice([0.0, 0.0, 0.0, 1.0, float("inf"), float("nan")]))
        gr, bo = float(rng.choice([2.0, 1.5, 1e10])), float(rng.choice([0.5, 0.25]))
        ts = torch.tensor([sc], dtype=torch.float32)
        tt = torch.tensor([tr], dtype=torch.int32)
        torch._amp_update_scale_(ts, tt, torch.tensor([fi], dtype=torch.float32), gr, bo, iv)
        got_sc, got_tr = orc.amp_update_scale(sc, tr, fi, gr, bo, iv)
        assert got_tr == int(tt.item()), (sc, tr, fi, gr, bo, iv)
        assert np.float32(got_sc).tobytes() == ts.numpy().tobytes(), (sc, tr, fi, gr, bo, iv, got_sc, ts)


def pin_any_nonfinite(orc):
    gen = torch.Generator().manual_seed(3)
    for dtype in (torch.bfloat16, torch.float16, torch.float32):
        x = torch.randn(1000, generator=gen).to(dtype)
        assert not orc.any_nonfinite(x)
        assert not orc.any_nonfinite(x[:0])
        for bad in (float("inf"), float("-inf"), float("nan")):
            y = x.clone()
            y[int(torch.randint(0, 1000, (1,), generator=gen))] = bad
            assert orc.any_nonfinite(y)
        big = torch.full((10,), 6.0e4 if dtype == torch.float16 else 3.0e38, dtype=torch.float32).to(dtype)
        assert not orc.any_nonfinite(big)  # large but finite


# ---- quantised reduce (page "aclnnQuantReduceScatter") -----------------------

def pin_decode8_all_patterns(orc):
    bits = np.arange(256, dtype=np.uint8)
    t = torch.from_numpy(bits.copy())
    for kind, want in ((0, t.view(torch.float8_e4m3fn).to(torch.float64)),
                       (1, t.view(torch.float8_e5m2).to(torch.float64)),
                       (2, t.view(torch.int8).to(torch.float64)),
                       (3, t.view(torch.float8_e8m0fnu).to(torch.float64))):
        got = orc.decode8(kind, bits)
        w = want.numpy()
        nan = np.isnan(w)
        assert np.array_equal(np.isnan(got), nan), kind
        assert np.array_equal(got[~nan], w[~nan]), kind


def _qr_case(case):
    W, rows, H = case["W"], case["rows"], case["H"]
    data = np.zeros((W, rows, H), np.int64)
    for w in range(W):
        data[w, 0, :] = case["data_fill"][w]
        data[w, 0, :4] = case["data_first4"][w]
    return W, rows, H, data.astype(np.int8).view(np.uint8) if data.min() < 0 else data.astype(np.uint8)


def pin_quant_reduce_golden(orc):
    g = _golden("quant_reduce.json")
    c = g["mx_e4m3"]
    W, rows, H, data = _qr_case(c)
    scales = np.array(c["scales"], np.uint8).reshape(W, rows, H // 32)
    out = orc.quant_reduce(data, scales, 0, 0)
    assert out[0, :4].tolist() == c["want_first4"] and (out[0, 4:] == c["want_fill"]).all()
    c = g["pergroup_int8"]
    W, rows, H, data = _qr_case(c)
    scales = np.array(c["scales"], np.float32).reshape(W, rows, H // 128)
    out = orc.quant_reduce(data, scales, 2, 1)
    assert out[0, :4].tolist() == c["want_first4"] and (out[0, 4:] == c["want_fill"]).all()


def pin_quant_reduce_single_rank_unit_scale(orc):
    # One rank, scale 1 (E8M0 127, or 1.0f): the reduce is just the decode.
    rng = np.random.default_rng(12)
    data = rng.integers(0, 256, (1, 5, 256), dtype=np.uint8)
    data[(data & 0x7F) == 0x7F] = 0  # no NaN codes
    for q in (0, 1):
        data_q = data.copy()
        if q == 1:
            data_q[(data_q & 0x7C) == 0x7C] = 0  # no inf/NaN codes
        out = orc.quant_reduce(data_q, np.full((1, 5, 8), 127, np.uint8), q, 0)
        assert np.array_equal(out, orc.decode8(q, data_q[0]))
        out = orc.quant_reduce(data_q, np.ones((1, 5, 2), np.float32), q, 1)
        assert np.array_equal(out, orc.decode8(q, data_q[0]))


def pin_quant_reduce_scale_locality(orc):
    # Every value 1.0 (E4M3 0x38, INT8 1) and one rank: each output is exactly
    # the scale of its own (row, group), 2^(e - 127) for E8M0.
    rng = np.random.default_rng(14)
    rows, H = 3, 512
    e = rng.integers(100, 150, (1, rows, H // 32), dtype=np.uint8)
    out = orc.quant_reduce(np.full((1, rows, H), 0x38, np.uint8), e, 0, 0)
    assert np.array_equal(out, np.repeat(2.0 ** (e[0].astype(np.float64) - 127), 32, axis=1))
    f = rng.standard_normal((1, rows, H // 128)).astype(np.float32)
    out = orc.quant_reduce(np.ones((1, rows, H), np.uint8), f, 2, 1)
    assert np.array_equal(out, np.repeat(f[0].astype(np.float64), 128, axis=1))


def pin_quant_reduce_linear_in_ranks(orc):
    # Doubling rank w's scales adds exactly rank w's contribution once more;
    # the rows and groups stay where they are.
    rng = np.random.default_rng(13)
    W, rows, H = 4, 6, 256
    data = rng.integers(0, 127, (W, rows, H), dtype=np.uint8)  # positive E4M3 codes
    scales = rng.integers(120, 135, (W, rows, H // 32), dtype=np.uint8)
    base = orc.quant_reduce(data, scales, 0, 0)
    for w in range(W):
        s2 = scales.copy()
        s2[w] += 1
        one = np.zeros_like(scales)
        one[w] = scales[w]
        only_w = orc.quant_reduce(np.where(np.arange(W)[:, None, None] == w, data, 0).astype(np.uint8),
                                  np.maximum(one, 1), 0, 0)
        assert np.allclose(orc.quant_reduce(data, s2, 0, 0), base + only_w, rtol=1e-15, atol=0)


def pin_quant_reduce_rejects_bad_modes(orc):
    d = np.zeros((2, 1, 64), np.uint8)
    for args in ((d, np.zeros((2, 1, 2), np.uint8), 2, 0),       # mx mode takes FLOAT8 only
                 (d, np.zeros((2, 1, 1), np.float32), 0, 1)):    # H not a multiple of 128
        try:
            orc.quant_reduce(*args)
        except OracleError:
            continue
        raise AssertionError("accepted")


# ---- block-scaled FP8 grouped product (mx operands) ---------------------------

def _mx_decode(codes, scales, qtype):
    """Exact values of mx-quantised rows by torch's own float8 decoders: codes [..., K],
    E8M0 scales [..., K/32]."""
    t = torch.from_numpy(np.ascontiguousarray(codes))
    v = t.view(torch.float8_e4m3fn if qtype == 0 else torch.float8_e5m2).to(torch.float64)
    s = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e8m0fnu).to(torch.float64)
    return (v * s.repeat_interleave(32, dim=-1)).numpy()


def _mx_random(rng, shape, qtype, lo=120, hi=134):
    """Random finite codes of a format and E8M0 scales in [lo, hi]."""
    finite = np.array([c for c in range(256) if (qtype == 0 and (c & 0x7F) != 0x7F)
                       or (qtype == 1 and (c & 0x7C) != 0x7C)], np.uint8)
    codes = finite[rng.integers(0, len(finite), shape)]
    scales = rng.integers(lo, hi + 1, shape[:-1] + (shape[-1] // 32,)).astype(np.uint8)
    return codes, scales


def pin_mx_grouped_matmul_golden(orc):
    g = _golden("mx_grouped_matmul.json")
    for q, key in ((0, "e4m3"), (1, "e5m2")):
        c = g[key]
        K = c["K"]
        a = np.repeat(np.array(c["a_codes"], np.uint8), 32)[None, :]
        sa = np.array(c["a_scales"], np.uint8)[None, :]
        w = np.stack([np.repeat(np.array(col, np.uint8), 32) for col in c["w_codes"]])[None]
        sw = np.array(c["w_scales"], np.uint8)[None]
        assert a.shape == (1, K)
        out = orc.mx_grouped_matmul([1], a, sa, w, sw, q, q)
        assert out[0].tolist() == c["want"], (key, out)


def pin_mx_grouped_matmul_numpy(orc):
    # Against numpy float64 products of operands decoded by torch.
    rng = np.random.default_rng(31)
    for q in (0, 1):
        e, K, N = 3, 96, 24
        gr = [5, 0, 9]
        a, sa = _mx_random(rng, (14, K), q)
        w, sw = _mx_random(rng, (e, N, K), q)
        got = orc.mx_grouped_matmul(gr, a, sa, w, sw, q, q)
        x = _mx_decode(a, sa, q)
        wv = _mx_decode(w, sw, q)
        expert = np.repeat(np.arange(e), gr)
        want = np.stack([x[i] @ wv[expert[i]].T for i in range(14)])
        assert np.allclose(got, want, rtol=1e-12, atol=1e-300), q


def pin_mx_scale_block_locality(orc):
    # Only block b of the row carries non-zero codes: the other blocks' scales
    # cannot matter, and one step of block b's scale doubles the result.
    K, N = 128, 4
    a = np.zeros((1, K), np.uint8)
    a[0, 64:96] = 0x38  # 1.0 in block 2
    sa = np.array([[100, 140, 127, 90]], np.uint8)
    w = np.full((1, N, K), 0x38, np.uint8)
    sw = np.full((1, N, K // 32), 127, np.uint8)
    base = orc.mx_grouped_matmul([1], a, sa, w, sw, 0, 0)
    assert (base == 32.0).all()
    sa2 = sa.copy()
    sa2[0, [0, 1, 3]] = [130, 110, 127]
    assert np.array_equal(orc.mx_grouped_matmul([1], a, sa2, w, sw, 0, 0), base)
    sa2[0, 2] = 128
    assert (orc.mx_grouped_matmul([1], a, sa2, w, sw, 0, 0) == 64.0).all()
    sw2 = sw.copy()
    sw2[0, 1, 2] = 125  # column 1, block 2: a quarter
    out = orc.mx_grouped_matmul([1], a, sa, w, sw2, 0, 0)
    assert out[0].tolist() == [32.0, 8.0, 32.0, 32.0]


def pin_mx_group_boundaries_scaled_identity(orc):
    # w[j][n][k] = 2^j * [k == n] (E4M3 1.0 with E8M0 scale 127 + j): row i of
    # group j gives 2^j * x[i][:N], exactly, across an empty group.
    rng = np.random.default_rng(32)
    K = N = 64
    gr = [3, 0, 4, 2]
    a, sa = _mx_random(rng, (9, K), 0, 124, 130)
    w = np.zeros((4, N, K), np.uint8)
    for n in range(N):
        w[:, n, n] = 0x38
    sw = np.repeat((127 + np.arange(4, dtype=np.uint8))[:, None, None], N, 1).repeat(K // 32, 2)
    got = orc.mx_grouped_matmul(gr, a, sa, w, sw, 0, 0)
    x = _mx_decode(a, sa, 0)
    expert = np.repeat(np.arange(4), gr)
    assert np.array_equal(got, x * (2.0 ** expert)[:, None])


def pin_mx_rows_subset_and_rejects(orc):
    rng = np.random.default_rng(33)
    a, sa = _mx_random(rng, (7, 64), 1)
    w, sw = _mx_random(rng, (2, 5, 64), 1)
    full = orc.mx_grouped_matmul([3, 4], a, sa, w, sw, 1, 1)
    rows = [6, 0, 3, 3]
    assert np.array_equal(orc.mx_grouped_matmul([3, 4], a, sa, w, sw, 1, 1, rows=rows), full[rows])
    for args in (([3, 3], a, sa, w, sw, 1, 1), ([3, 4], a, sa, w, sw, 2, 1)):
        try:
            orc.mx_grouped_matmul(*args)
        except OracleError:
            continue
        raise AssertionError(f"accepted {args[0]}, qa={args[5]}")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
