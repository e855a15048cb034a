// Permute: ataOut (rank-major) -> expert-major rows, a pure row gather.
//
// "aclnnAlltoAllvGroupedMatMul", Formula: permuteOut = Permute(ataOut).
// One warp moves one row at a time with 16-byte vector loads and stores
// (coalesced across the warp); each CTA first rebuilds the segment table from
// recvCounts in shared memory (one warp, a few hundred cycles).
#include "kernels.h"
#include "plan.cuh"

namespace a2av {

namespace {

constexpr int kPermuteThreads = 256;
constexpr int kPermuteWarps = kPermuteThreads / 32;

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
    __shared__ int ok;
    // A GEMM launched after this kernel with programmatic dependent launch
    // may start now: it waits for this grid's completion before it reads
    // any row this kernel writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0) {
        bool good = build_segment_table(recvCounts, W, e, A, table, lane);
        if (lane == 0) {
            ok = good;
            if (blockIdx.x == 0) {
                if (write_status) *status = good ? 0 : kStatusBadCounts;
                else if (!good) atomicOr(status, kStatusBadCounts);
            }
        }
    }
    __syncthreads();
    if (!ok) return;

    const int vpr = H1 / 8;  // 16-byte vectors per row
    const int nwarps = gridDim.x * kPermuteWarps;
    for (int d = blockIdx.x * kPermuteWarps + warp; d < A; d += nwarps) {
        const int seg = segment_of(table, W, e, d);
        if (only_straddling) {
            // Copy only the rows of 128-row halves that the GEMM cannot read
            // in place (see half_in_one_segment).
            const int j = seg / W;
            const int g0 = table.dst[j * W], g1 = table.dst[(j + 1) * W];
            const int first = g0 + (d - g0) / kHalfRows * kHalfRows;
            if (half_in_one_segment(table, W, e, first, g1)) continue;
        }
        const int s = source_row_in(table, W, e, seg, d);
        const uint4 *in = src + static_cast<size_t>(s) * vpr;
        uint4 *out = dst + static_cast<size_t>(d) * vpr;
        int v = lane;
        for (; v + 96 < vpr; v += 128) {
            uint4 a = ld_stream(in + v), b = ld_stream(in + v + 32), c = ld_stream(in + v + 64),
                  f = ld_stream(in + v + 96);
            out[v] = a;
            out[v + 32] = b;
            out[v + 64] = c;
            out[v + 96] = f;
        }
        for (; v < vpr; v += 32) out[v] = ld_stream(in + v);
    }
}

}  // namespace

cudaError_t launch_permute(const PermuteLaunch &p, int num_sms, cudaStream_t stream) {
    int blocks = (p.A + kPermuteWarps - 1) / kPermuteWarps;
    const int cap = num_sms * (p.blocks_per_sm > 0 ? p.blocks_per_sm : 2048 / kPermuteThreads);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    permute_rows_kernel<<<blocks, kPermuteThreads, 0, stream>>>(
        p.recvCounts, p.W, p.e, p.A, p.H1, static_cast<const uint4 *>(p.ataOut),
        static_cast<uint4 *>(p.dst), p.status, p.write_status, p.only_straddling);
    return cudaGetLastError();
}

}  // namespace a2av
