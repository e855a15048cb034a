"""Seeded synthetic inputs for the AlltoAllv + Permute + GroupedMatMul hot path.

This module only draws inputs: the received-count vector ``recvCounts`` of
one simulated rank and the tensors ``ataOut``, ``gmmWeight``, ``mmX`` and
``mmWeight``.  It holds none of the operator's arithmetic (no offsets, no
permutation, no products), so both the CUDA path and the CPU oracle can take
their inputs from it without sharing any of the computation.

Routing model (the pages give the operator, not its inputs; these are the
synthetic stand-ins).  Rank 0 of an expert-parallel domain of ``W`` ranks owns
global experts ``0 .. e-1`` (global id = rank * e + j).  Each source rank ``w``
routes ``tokens_per_source`` tokens, each to its top-``K`` of ``E = W * e``
global experts, and ``recvCounts[w * e + j]`` is how many of those selections
hit local expert ``j`` ("Shape variables": A is the sum of recvCounts, and the
A's of all ranks add up to the BSK's of all ranks, so every selection lands on
exactly one rank).

Random streams: ``numpy.random.default_rng([seed, stream, chunk])`` with
stream 0 for routing, 1 for ataOut, 2 for gmmWeight, 3 for mmX, 4 for
mmWeight.  Tensors are drawn in float32 in fixed 4 Mi-element chunks (so the
values do not depend on the thread count) and rounded to bf16/fp16 by torch
(round to nearest even).  Both sides consume the rounded tensors.
"""

from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

_CHUNK = 1 << 22

STREAM_ROUTING = 0
STREAM_ATAOUT = 1
STREAM_GMM_WEIGHT = 2
STREAM_MMX = 3
STREAM_MM_WEIGHT = 4
STREAM_GMMX = 7  # a source rank's rows before the AlltoAllv


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: the shape of one rank's share of a MoE layer."""

    name: str
    W: int                      # ranks in the expert-parallel domain
    e: int                      # local experts on this rank
    H1: int                     # routed hidden size (GEMM K)
    N1: int                     # routed output width (GEMM N)
    dtype: str                  # "bf16" or "fp16"
    routing: str                # "uniform", "normal", "zipf"
    tokens_per_source: int = 0  # tokens each source routes (BS of that rank)
    topk: int = 0               # K of top-K
    A_total: int = 0            # only for routing == "uniform"
    bias_std: float = 0.0       # per-expert logit bias (normal routing)
    zipf_s: float = 0.0         # popularity exponent (zipf routing)
    empty_fraction: float = 0.0  # share of (w, j) segments forced to 0 rows
    BS: int = 0                 # shared-expert rows (0: no shared expert)
    H2: int = 0
    N2: int = 0
    act_scale_by_h1: bool = False  # ataOut ~ N(0,1)/sqrt(H1) instead of N(0,1)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "fp16": torch.float16}[self.dtype]


# The five workloads.  Names say what each is, with its sizes.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_w2e2_h256_n128", W=2, e=2, H1=256, N1=128, dtype="bf16",
                 routing="uniform", A_total=256, act_scale_by_h1=True),
        Workload("w8e4_h4096_n1024_shared2048", W=8, e=4, H1=4096, N1=1024,
                 dtype="bf16", routing="normal", tokens_per_source=2048, topk=8,
                 BS=2048, H2=4096, N2=1024),
        Workload("dsv3_w32e8_h7168_n4096_shared4096", W=32, e=8, H1=7168,
                 N1=4096, dtype="bf16", routing="normal", tokens_per_source=4096,
                 topk=8, bias_std=0.5, BS=4096, H2=7168, N2=4096),
        Workload("skew_w8e32_h4096_n1536_fp16", W=8, e=32, H1=4096, N1=1536,
                 dtype="fp16", routing="zipf", tokens_per_source=4096, topk=8,
                 zipf_s=1.2, empty_fraction=0.2),
        Workload("large_a_w16e16_h2048_n1408_shared16384", W=16, e=16, H1=2048,
                 N1=1408, dtype="bf16", routing="normal", tokens_per_source=16384,
                 topk=4, BS=16384, H2=2048, N2=5632),
        # The large-A text quotes A of about 262K, which is W * BS; top-4 over
        # 256 experts gives each rank about BS * K = 65.5K.  This variant
        # routes 4 * BS tokens per source so that A lands near 262K.
        Workload("large_a262k_w16e16_h2048_n1408_shared16384", W=16, e=16,
                 H1=2048, N1=1408, dtype="bf16", routing="normal",
                 tokens_per_source=4 * 16384, topk=4, BS=16384, H2=2048,
                 N2=5632),
    ]
}

SMALL = "tiny_w2e2_h256_n128"
W8E4 = "w8e4_h4096_n1024_shared2048"
# The bench's default: the largest workload that fits one GPU by FLOPs (the
# DeepSeek-V3-like layer, about 2.2 TFLOP per call).
HEADLINE = "dsv3_w32e8_h7168_n4096_shared4096"


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, stream, chunk])


def normal_f32(n: int, seed: int, stream: int) -> np.ndarray:
    """n standard normals in float32, drawn in fixed chunks on a thread pool."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(i: int) -> None:
        s = i * _CHUNK
        t = min(n, s + _CHUNK)
        _rng(seed, stream, i).standard_normal(t - s, dtype=np.float32, out=out[s:t])

    if nchunks <= 1:
        if n:
            fill(0)
    else:
        workers = min(nchunks, os.cpu_count() or 1)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def rounded(x: np.ndarray, shape, dtype: torch.dtype) -> torch.Tensor:
    """float32 values rounded to a 16-bit float type (round to nearest even)."""
    return torch.from_numpy(x).reshape(shape).to(dtype)


def _topk_counts(scores: np.ndarray, k: int, lo: int, e: int) -> np.ndarray:
    """Hits on experts lo..lo+e-1 of each token's top-k (scores: [tokens, E])."""
    top = np.argpartition(-scores, k - 1, axis=1)[:, :k]
    return np.bincount(top.ravel(), minlength=scores.shape[1])[lo:lo + e]


def recv_counts(wl: Workload, seed: int = 0, rank: int = 0) -> np.ndarray:
    """recvCounts of one rank, int32, index w * e + j (source rank major).

    Every rank sees the same routing draw; rank r owns global experts
    r*e .. r*e + e - 1.
    """
    W, e = wl.W, wl.e
    E = W * e
    lo = rank * e
    rng = _rng(seed, STREAM_ROUTING)
    if wl.routing == "uniform":
        rc = _rng(seed, STREAM_ROUTING, rank).multinomial(wl.A_total, [1.0 / E] * E)
        return rc.astype(np.int32)

    rc = np.zeros(E, dtype=np.int64)
    if wl.routing == "normal":
        rc[:] = routing_counts(wl, seed)[:, lo:lo + e].reshape(-1)
    elif wl.routing == "zipf":
        # Popularity p_x proportional to rank(x)^-s over a seeded ranking of
        # the E experts; each token samples K distinct experts with
        # probability proportional to p (Gumbel-top-K of log p).
        order = rng.permutation(E)
        popularity_rank = np.empty(E, dtype=np.int64)
        popularity_rank[order] = np.arange(1, E + 1)
        logp = -wl.zipf_s * np.log(popularity_rank.astype(np.float64))
        for w in range(W):
            g = rng.gumbel(size=(wl.tokens_per_source, E))
            rc[w * e:(w + 1) * e] = _topk_counts(logp[None, :] + g, wl.topk, lo, e)
        # Force round(frac * E) empty segments: first the least popular local
        # experts for every source (whole empty GEMM groups), then single
        # (w, j) segments inside experts that keep rows.
        n_empty = int(round(wl.empty_fraction * E))
        local_by_pop = np.argsort(-logp[lo:lo + e], kind="stable")[::-1]  # least popular first
        whole = n_empty // W
        for j in local_by_pop[:whole]:
            rc[j::e] = 0
        rest = n_empty - whole * W
        keep = [w * e + j for j in sorted(local_by_pop[whole:]) for w in range(W)]
        for idx in rng.choice(np.array(keep), size=rest, replace=False):
            rc[idx] = 0
    else:
        raise ValueError(wl.routing)
    return rc.astype(np.int32)


def routing_counts(wl: Workload, seed: int = 0) -> np.ndarray:
    """[W, W*e] int64: how many of source rank w's top-K selections hit global
    expert g, for the "normal" routing model (one draw shared by all ranks)."""
    if wl.routing != "normal":
        raise ValueError("routing_counts models the sender side of normal routing only")
    W, E = wl.W, wl.W * wl.e
    rng = _rng(seed, STREAM_ROUTING)
    bias = (rng.standard_normal(E) * wl.bias_std) if wl.bias_std else np.zeros(E)
    out = np.zeros((W, E), dtype=np.int64)
    for w in range(W):
        logits = rng.standard_normal((wl.tokens_per_source, E), dtype=np.float32)
        logits += bias.astype(np.float32)
        out[w] = _topk_counts(logits, wl.topk, 0, E)
    return out


def send_counts(wl: Workload, seed: int = 0, rank: int = 0) -> np.ndarray:
    """sendCounts of source rank `rank`: int32 [W*e], entry g = rows it sends to
    global expert g (owned by rank g // e as its local expert g % e)."""
    return routing_counts(wl, seed)[rank].astype(np.int32)


def make_gmmX(wl: Workload, seed: int = 0, rank: int = 0) -> tuple[torch.Tensor, np.ndarray]:
    """(gmmX, sendCounts) of one source rank: [sum(sendCounts), H1] N(0,1) rows,
    grouped by destination global expert in ascending order, drawn from seed + rank."""
    sc = send_counts(wl, seed, rank)
    n = int(sc.astype(np.int64).sum())
    x = rounded(normal_f32(n * wl.H1, seed + rank, STREAM_GMMX), (n, wl.H1), wl.torch_dtype)
    return x, sc


@dataclasses.dataclass
class Inputs:
    wl: Workload
    recvCounts: np.ndarray          # int32 [W*e]
    ataOut: torch.Tensor            # [A, H1] 16-bit, CPU
    gmmWeight: torch.Tensor         # [e, H1, N1]
    mmX: torch.Tensor | None        # [BS, H2]
    mmWeight: torch.Tensor | None   # [H2, N2]

    @property
    def A(self) -> int:
        return int(self.ataOut.shape[0])


def make_inputs(wl: Workload, seed: int = 0, rank: int = 0) -> Inputs:
    """All inputs of one workload for one rank, as CPU tensors (see module
    docstring).  Tensor values are drawn from seed + rank."""
    rc = recv_counts(wl, seed, rank)
    seed = seed + rank
    A = int(rc.astype(np.int64).sum())
    dt = wl.torch_dtype
    act = normal_f32(A * wl.H1, seed, STREAM_ATAOUT)
    if wl.act_scale_by_h1:
        act *= np.float32(1.0 / math.sqrt(wl.H1))
    ata = rounded(act, (A, wl.H1), dt)
    del act
    wt = normal_f32(wl.e * wl.H1 * wl.N1, seed, STREAM_GMM_WEIGHT)
    wt *= np.float32(1.0 / math.sqrt(wl.H1))
    gw = rounded(wt, (wl.e, wl.H1, wl.N1), dt)
    del wt
    mmX = mmW = None
    if wl.BS:
        x = normal_f32(wl.BS * wl.H2, seed, STREAM_MMX)
        mmX = rounded(x, (wl.BS, wl.H2), dt)
        wm = normal_f32(wl.H2 * wl.N2, seed, STREAM_MM_WEIGHT)
        wm *= np.float32(1.0 / math.sqrt(wl.H2))
        mmW = rounded(wm, (wl.H2, wl.N2), dt)
    return Inputs(wl, rc, ata, gw, mmX, mmW)


def custom_inputs(W: int, e: int, H1: int, N1: int, rc, dtype: str = "bf16",
                  BS: int = 0, H2: int = 0, N2: int = 0, seed: int = 0) -> Inputs:
    """Inputs for an explicit count vector (edge cases in the tests)."""
    wl = Workload(f"custom_w{W}e{e}_h{H1}_n{N1}", W=W, e=e, H1=H1, N1=N1,
                  dtype=dtype, routing="given", BS=BS, H2=H2, N2=N2)
    rc = np.asarray(rc, dtype=np.int32)
    assert rc.shape == (W * e,)
    A = int(rc.astype(np.int64).sum())
    dt = wl.torch_dtype
    ata = rounded(normal_f32(A * H1, seed, STREAM_ATAOUT), (A, H1), dt)
    wt = normal_f32(e * H1 * N1, seed, STREAM_GMM_WEIGHT) * np.float32(1.0 / math.sqrt(H1))
    gw = rounded(wt, (e, H1, N1), dt)
    mmX = mmW = None
    if BS:
        mmX = rounded(normal_f32(BS * H2, seed, STREAM_MMX), (BS, H2), dt)
        wm = normal_f32(H2 * N2, seed, STREAM_MM_WEIGHT) * np.float32(1.0 / math.sqrt(H2))
        mmW = rounded(wm, (H2, N2), dt)
    return Inputs(wl, rc, ata, gw, mmX, mmW)


def random_counts(W: int, e: int, A: int, seed: int, zero_prob: float = 0.0) -> np.ndarray:
    """A seeded count vector summing to A, with some segments forced empty."""
    rng = _rng(seed, STREAM_ROUTING, 1)
    E = W * e
    live = rng.random(E) >= zero_prob
    if not live.any() and A:
        live[rng.integers(E)] = True
    p = np.where(live, rng.random(E) + 0.05, 0.0)
    rc = np.zeros(E, dtype=np.int64)
    if A:
        rc = rng.multinomial(A, p / p.sum())
    return rc.astype(np.int32)


# --- Quantised reduce ("aclnnQuantReduceScatter" page) -----------------------
#
# After the AllToAll, a rank holds from each of W source ranks `rows` rows of
# H 8-bit codes plus their scales.  The page fixes the formats and limits
# (W in {2, 4, 8}, H a multiple of 128 in [1024, 8192]) but not the values:
# codes are drawn uniformly from the format's finite codes, and scales are
# powers of two (E8M0 codes, mx mode) or float32 2^u with u uniform (per-128
# groups), both over the same exponent range.

STREAM_QDATA = 5
STREAM_QSCALES = 6

QTYPE_NAMES = ("e4m3fn", "e5m2", "int8")
QMODE_NAMES = ("mx", "group128")


@dataclasses.dataclass(frozen=True)
class QuantReduceWorkload:
    name: str
    W: int
    rows: int   # rows received from each source rank (BS / W)
    H: int
    qtype: str  # "e4m3fn", "e5m2" or "int8"
    mode: str   # "mx" (E8M0 scales per 32) or "group128" (float32 scales per 128)


# BS = 12288 tokens of H = 7168 on W = 8 ranks: x is 88 MB per rank, inside the
# page's default 200 MB communication buffer (HCCL_BUFFSIZE >= 2 (x + scales + 1) MB).
QREDUCE_WORKLOADS = {
    w.name: w
    for w in (
        QuantReduceWorkload("qreduce_mx_e4m3_w8_rows1536_h7168", 8, 1536, 7168, "e4m3fn", "mx"),
        QuantReduceWorkload("qreduce_g128_int8_w8_rows1536_h7168", 8, 1536, 7168, "int8", "group128"),
        QuantReduceWorkload("qreduce_mx_e5m2_w4_rows2048_h4096", 4, 2048, 4096, "e5m2", "mx"),
        QuantReduceWorkload("qreduce_mx_e5m2_w2_rows64_h1024", 2, 64, 1024, "e5m2", "mx"),
    )
}
QREDUCE_HEADLINE = "qreduce_mx_e4m3_w8_rows1536_h7168"


def finite_codes(qtype: str) -> np.ndarray:
    """The 8-bit codes of a format that encode finite numbers (by bit pattern only)."""
    codes = np.arange(256, dtype=np.uint8)
    if qtype == "e4m3fn":
        return codes[(codes & 0x7F) != 0x7F]            # S.1111.111 is NaN
    if qtype == "e5m2":
        return codes[(codes & 0x7C) != 0x7C]            # exponent field all ones: inf/NaN
    return codes


def quant_reduce_inputs(W: int, rows: int, H: int, qtype: str, mode: str, seed: int = 0,
                        exp_range=(-10, 6)) -> tuple[torch.Tensor, torch.Tensor]:
    """(data uint8 [W, rows, H], scales) on the CPU: E8M0 codes uint8 [W, rows, H/32] for
    mode "mx", float32 [W, rows, H/128] for "group128"; scale exponents in exp_range."""
    n = W * rows * H
    allowed = finite_codes(qtype)
    data = np.empty(n, dtype=np.uint8)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(i: int) -> None:
        s, t = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        data[s:t] = allowed[_rng(seed, STREAM_QDATA, i).integers(0, len(allowed), t - s)]

    with ThreadPoolExecutor(max(1, min(nchunks, os.cpu_count() or 1))) as ex:
        list(ex.map(fill, range(nchunks)))
    lo, hi = exp_range
    rng = _rng(seed, STREAM_QSCALES)
    if mode == "mx":
        sc = (rng.integers(lo, hi + 1, W * rows * (H // 32)) + 127).astype(np.uint8).reshape(W, rows, H // 32)
    else:
        sc = np.exp2(rng.uniform(lo, hi, W * rows * (H // 128))).astype(np.float32).reshape(W, rows, H // 128)
    return torch.from_numpy(data.reshape(W, rows, H)), torch.from_numpy(sc)


# --- Block-scaled FP8 (mx) operands --------------------------------------------
#
# The mx variant of a workload draws the same float32 tensors as make_inputs
# and quantises each 32-element block along K the OCP MX way: the block's
# E8M0 scale is 2^(floor(log2 amax) - emax) with emax the format's largest
# exponent (8 for E4M3FN, 15 for E5M2); the codes are the scaled values
# rounded to the format by torch's own float8 cast (saturating at the largest
# finite value).  Weights are stored K-contiguous per output column: [e, N1, H1].

_F8 = {"e4m3fn": (torch.float8_e4m3fn, 8, 448.0), "e5m2": (torch.float8_e5m2, 15, 57344.0)}


def mx_quantize(x: torch.Tensor, qtype: str) -> tuple[torch.Tensor, torch.Tensor]:
    """float32 [..., K] (K % 32 == 0) -> (uint8 codes [..., K], uint8 E8M0 scales [..., K/32])."""
    f8, emax, fmax = _F8[qtype]
    xb = x.reshape(*x.shape[:-1], x.shape[-1] // 32, 32)
    amax = xb.abs().amax(-1)
    e = torch.where(amax > 0, torch.floor(torch.log2(amax)), torch.full_like(amax, -127.0)) - emax
    e = e.clamp(-127, 127)
    codes = (xb / torch.exp2(e)[..., None]).clamp(-fmax, fmax).to(f8).view(torch.uint8)
    return codes.reshape(x.shape), (e + 127).to(torch.uint8)


@dataclasses.dataclass
class MxInputs:
    wl: Workload
    qtype: str
    recvCounts: np.ndarray           # int32 [W*e]
    ataOut_q: torch.Tensor           # [A, H1] codes
    ataOut_s: torch.Tensor           # [A, H1/32] E8M0
    gmmWeight_q: torch.Tensor        # [e, N1, H1]
    gmmWeight_s: torch.Tensor        # [e, N1, H1/32]
    mmX_q: torch.Tensor | None = None
    mmX_s: torch.Tensor | None = None
    mmWeight_q: torch.Tensor | None = None  # [N2, H2]
    mmWeight_s: torch.Tensor | None = None

    @property
    def A(self) -> int:
        return int(self.ataOut_q.shape[0])


def make_mx_inputs(wl: Workload, seed: int = 0, rank: int = 0, qtype: str = "e4m3fn",
                   recvCounts=None) -> MxInputs:
    """The mx operands of one rank (CPU tensors): the float32 draws of make_inputs, quantised."""
    rc = recv_counts(wl, seed, rank) if recvCounts is None else np.asarray(recvCounts, np.int32)
    seed = seed + rank
    A = int(rc.astype(np.int64).sum())
    act = torch.from_numpy(normal_f32(A * wl.H1, seed, STREAM_ATAOUT)).reshape(A, wl.H1)
    aq, as_ = mx_quantize(act, qtype)
    wt = torch.from_numpy(normal_f32(wl.e * wl.H1 * wl.N1, seed, STREAM_GMM_WEIGHT)).reshape(wl.e, wl.H1, wl.N1)
    wq, ws = mx_quantize(wt.transpose(1, 2).contiguous() * (1.0 / math.sqrt(wl.H1)), qtype)
    out = MxInputs(wl, qtype, rc, aq, as_, wq, ws)
    if wl.BS:
        x = torch.from_numpy(normal_f32(wl.BS * wl.H2, seed, STREAM_MMX)).reshape(wl.BS, wl.H2)
        out.mmX_q, out.mmX_s = mx_quantize(x, qtype)
        wm = torch.from_numpy(normal_f32(wl.H2 * wl.N2, seed, STREAM_MM_WEIGHT)).reshape(wl.H2, wl.N2)
        out.mmWeight_q, out.mmWeight_s = mx_quantize(wm.t().contiguous() * (1.0 / math.sqrt(wl.H2)), qtype)
    return out
