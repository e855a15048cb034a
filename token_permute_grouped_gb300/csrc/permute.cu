// Permute: ataOut (rank-major) -> expert-major rows, a pure row gather.
//
// "aclnnAlltoAllvGroupedMatMul", Formula: permuteOut = Permute(ataOut).
// A warp moves one 2 KB piece of a row at a time with 16-byte vector loads
// and stores (coalesced across the warp); each CTA first rebuilds the segment table from
// recvCounts in shared memory (one warp, a few hundred cycles).
#include <algorithm>

#include "kernels.h"
#include "plan.cuh"

namespace a2av {

namespace {

constexpr int kPermuteThreads = 256;
constexpr int kPermuteWarps = kPermuteThreads / 32;
constexpr int kPieceVecs = 4;  // 16-byte vectors per lane in one work item (2 KB per warp)

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kPermuteThreads)
    permute_rows_kernel(const int32_t *__restrict__ recvCounts, int W, int e, int A, int H1,
                        const uint4 *__restrict__ src, uint4 *__restrict__ dst, int32_t *status,
                        int write_status, int only_straddling) {
    __shared__ SegmentTable table;
    __shared__ StagedHalves halves;
    __shared__ int ok;
    // The first kernel of a call clears the status word before the GEMM
    // behind it can start, so that later kernels only ever set bits in it
    // (atomicOr) and none of their bits is lost to this store.
    if (write_status && blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            *status = 0;
            __threadfence();
        }
        __syncthreads();
    }
    // A GEMM launched after this kernel with programmatic dependent launch
    // may start now: it waits for this grid's completion before it reads
    // any row this kernel writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0) {
        bool good = build_segment_table(recvCounts, W, e, A, table, lane);
        if (lane == 0) {
            ok = good;
            if (blockIdx.x == 0 && !good) atomicOr(status, kStatusBadCounts);
        }
    }
    __syncthreads();
    if (!ok) return;

    // Work items are pieces of a row (kPieceVecs 16-byte vectors per lane, all
    // loaded before any is stored): one memory round trip per item, and the
    // rows of a call spread over every warp of the grid.
    const int vpr = H1 / 8;  // 16-byte vectors per row
    const int ppr = (vpr + 32 * kPieceVecs - 1) / (32 * kPieceVecs);
    const int nwarps = gridDim.x * kPermuteWarps;
    const int gw = blockIdx.x * kPermuteWarps + warp;
    const auto copy_piece = [&](int d, int seg, int piece) {
        const int v0 = piece * 32 * kPieceVecs + lane;
        const int32_t s_row = source_row_in(table, W, e, seg, d);
        if (!in_bounds(seg >= 0 && seg < W * e && d >= 0 && d < A && s_row >= 0 && s_row < A, status)) return;
        const uint4 *in = src + static_cast<size_t>(s_row) * vpr;
        uint4 *out = dst + static_cast<size_t>(d) * vpr;
        uint4 r[kPieceVecs];
#pragma unroll
        for (int k = 0; k < kPieceVecs; ++k)
            if (v0 + 32 * k < vpr) r[k] = ld_stream(in + v0 + 32 * k);
#pragma unroll
        for (int k = 0; k < kPieceVecs; ++k)
            if (v0 + 32 * k < vpr) out[v0 + 32 * k] = r[k];
    };
    int listed = -1;
    if (only_straddling) {
        list_staged_halves(table, W, e, halves);
        listed = halves.n;
    }
    if (listed >= 0) {
        // Only the rows of the halves the GEMM cannot read in place.
        const int per_half = kHalfRows * ppr;
        for (int i = gw; i < listed * per_half; i += nwarps) {
            const int hi = i / per_half, rem = i - hi * per_half;
            const int r = rem / ppr;
            const int2 span = halves.span[hi];
            const int d = span.x + r;
            if (d < span.y) copy_piece(d, segment_of(table, W, e, d), rem - r * ppr);
        }
    } else {
        const int64_t items = static_cast<int64_t>(A) * ppr;
        for (int64_t i = gw; i < items; i += nwarps) {
            const int d = static_cast<int>(i / ppr);
            const int seg = segment_of(table, W, e, d);
            if (only_straddling) {
                // More staged halves than the list holds (not reached: see
                // kMaxStagedHalves): test each row's half.
                const int j = seg / W;
                const int g0 = table.dst[j * W], g1 = table.dst[(j + 1) * W];
                if (half_in_one_segment(table, W, e, g0 + (d - g0) / kHalfRows * kHalfRows, g1)) continue;
            }
            copy_piece(d, seg, static_cast<int>(i - static_cast<int64_t>(d) * ppr));
        }
    }
}

// Blocks of the permute kernel resident on one SM at once (per device, queried once).
int permute_blocks_per_sm() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, permute_rows_kernel, kPermuteThreads, 0) !=
            cudaSuccess)
            return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace

cudaError_t launch_permute(const PermuteLaunch &p, int num_sms, cudaStream_t stream) {
    int blocks = (p.A + kPermuteWarps - 1) / kPermuteWarps;
    // At most the blocks that are resident at once, so that none waits for a
    // second wave.
    const int resident = permute_blocks_per_sm();
    if (resident <= 0) return cudaErrorUnknown;
    const int cap = num_sms * (p.blocks_per_sm > 0 ? std::min<int>(p.blocks_per_sm, resident) : resident);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    permute_rows_kernel<<<blocks, kPermuteThreads, 0, stream>>>(
        p.recvCounts, p.W, p.e, p.A, p.H1, static_cast<const uint4 *>(p.ataOut),
        static_cast<uint4 *>(p.dst), p.status, p.write_status, p.only_straddling);
    return cudaGetLastError();
}

}  // namespace a2av
