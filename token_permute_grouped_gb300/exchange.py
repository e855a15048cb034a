"""The AlltoAllv in front of the hot path, over torch.distributed (NCCL on GPUs).

"aclnnAlltoAllvGroupedMatMul" page, Formula: ataOut = AlltoAllv(gmmX), then
permuteOut = Permute(ataOut), gmmY = permuteOut x gmmWeight, and, in parallel,
mmY = mmX x mmWeight.  Expert-parallel layout: rank r owns global experts
r*e .. r*e + e - 1 ("Shape variables": e local experts, W*e global ones).

Each source rank holds gmmX [BSK, H1] with its rows grouped by destination
global expert in ascending order, and sendCounts [W*e] (rows per global
expert).  The exchange is two collectives:

1. the counts: an all-to-all of e int32 per rank pair, which gives
   recvCounts[w*e + j] = sendCounts_w[r*e + j] on rank r;
2. the rows: an all-to-all-v with per-rank splits summed from those counts.
   Rank r receives source 0's rows first, then source 1's, ...; within a
   source they keep the sender's order (local expert ascending).  That is
   the rank-major ataOut that a2av_gmm_run takes.

The split sizes of step 2 must be known on the host, so step 1 is followed
by one device-to-host copy of the counts.  The collectives move bytes only;
the permute and both GEMMs run in the library's kernels (binding.Plan).

`layer` runs the exchange and then the hot path; optionally the shared
expert, which does not depend on the exchange, runs while the rows are in
flight.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding


def exchange_counts(sendCounts: torch.Tensor, e: int, group=None) -> torch.Tensor:
    """recvCounts [W*e] int32 from every rank's sendCounts [W*e] int32 (same device as the group's)."""
    W = dist.get_world_size(group)
    if sendCounts.dtype != torch.int32 or sendCounts.numel() != W * e:
        raise ValueError(f"sendCounts must be int32 [{W * e}]")
    recv = torch.empty_like(sendCounts)
    dist.all_to_all_single(recv, sendCounts.contiguous(), group=group)
    return recv


def alltoallv(gmmX: torch.Tensor, sendCounts: torch.Tensor, e: int, group=None,
              recvCounts: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """(ataOut [A, H1], recvCounts [W*e] int32): the AlltoAllv of gmmX.

    gmmX rows must be grouped by destination global expert, ascending, with
    sendCounts[g] rows for expert g.  recvCounts may be passed if already
    exchanged."""
    W = dist.get_world_size(group)
    if gmmX.dim() != 2:
        raise ValueError("gmmX must be [BSK, H1]")
    if recvCounts is None:
        recvCounts = exchange_counts(sendCounts, e, group)
    both = torch.stack([sendCounts, recvCounts]).cpu().to(torch.int64).reshape(2, W, e).sum(2)
    if (both < 0).any():
        raise ValueError("negative counts")
    in_splits, out_splits = both[0].tolist(), both[1].tolist()
    if sum(in_splits) != gmmX.shape[0]:
        raise ValueError(f"sendCounts sum to {sum(in_splits)}, gmmX has {gmmX.shape[0]} rows")
    ataOut = torch.empty(sum(out_splits), gmmX.shape[1], dtype=gmmX.dtype, device=gmmX.device)
    dist.all_to_all_single(ataOut, gmmX.contiguous(), out_splits, in_splits, group=group)
    return ataOut, recvCounts


def layer(gmmX: torch.Tensor, sendCounts: torch.Tensor, gmmWeight: torch.Tensor,
          mmX: torch.Tensor | None = None, mmWeight: torch.Tensor | None = None, group=None,
          want_permute_out: bool = False, overlap_shared: bool = False, path: str = "default",
          tiles: str = "default"):
    """The whole operator on this rank: AlltoAllv, then Permute + GroupedMatMul, and the
    shared-expert MatMul.  Returns (gmmY, mmY, permuteOut, ataOut, recvCounts).

    By default the shared expert runs with the routed experts after the
    exchange (one launch of the persistent kernel).  With overlap_shared it
    runs on the current stream while the row exchange runs on a side stream.
    The persistent kernel gives each CTA a fixed share of the tiles, so CTAs
    that wait for SMs held by the exchange's copy kernel finish late; on one
    GB300 that made the step twice as long (0.77 vs 0.38 ms on the
    8-rank-by-4-expert workload), so overlap is off by default."""
    e, H1, N1 = gmmWeight.shape
    W = dist.get_world_size(group)
    dev = gmmX.device
    BS = mmX.shape[0] if mmX is not None else 0
    H2 = mmX.shape[1] if mmX is not None else 0
    N2 = mmWeight.shape[1] if mmWeight is not None else 0
    compute = torch.cuda.current_stream(dev)
    recvCounts = exchange_counts(sendCounts, e, group)
    mmY = None
    if overlap_shared and BS:
        side = torch.cuda.Stream(dev)
        side.wait_stream(compute)
        with torch.cuda.stream(side):
            ataOut, recvCounts = alltoallv(gmmX, sendCounts, e, group, recvCounts)
        # The shared expert alone while the rows are in flight: a call with
        # A = 0 rows (and counts that sum to 0).
        shared = binding.Plan(W, e, 0, H1, N1, BS, H2, N2, gmmX.dtype, path=path, device=dev, tiles=tiles)
        no_rows = torch.zeros(W * e, dtype=torch.int32, device=dev)
        _, mmY, _ = shared.run(None, no_rows, gmmWeight, mmX, mmWeight, stream=compute)
        compute.wait_stream(side)
        ataOut.record_stream(compute)
        BS = H2 = N2 = 0
        mmX = mmWeight = None
    else:
        ataOut, recvCounts = alltoallv(gmmX, sendCounts, e, group, recvCounts)
    plan = binding.Plan(W, e, ataOut.shape[0], H1, N1, BS, H2, N2, gmmX.dtype,
                        want_permute_out=want_permute_out, path=path, device=dev, tiles=tiles)
    gmmY, mmY2, permuteOut = plan.run(ataOut, recvCounts, gmmWeight, mmX, mmWeight, stream=compute)
    return gmmY, (mmY if mmY is not None else mmY2), permuteOut, ataOut, recvCounts
