// Scan step: offsets of the (source rank, local expert) segments, computed on
// the device from recvCounts by one warp, into shared memory.
//
// "aclnnAlltoAllvGroupedMatMul", Formula: permuteOut = Permute(ataOut).
// ataOut is rank-major (segment w*e + j holds recvCounts[w*e + j] rows);
// permuteOut is expert-major (segment order j*W + w, arrival order kept
// inside each expert).  "Shape variables": A is the sum of recvCounts.
#pragma once

#include <cstdint>

namespace a2av {

constexpr int kMaxSegments = 256;  // W * e <= 256
constexpr int kMaxExperts = 32;    // e <= 32

// Device status word bits (written into the workspace).
constexpr int32_t kStatusBadCounts = 1;    // a negative count, or sum != A
constexpr int32_t kStatusTimeout = 2;      // a pipeline wait gave up
constexpr int32_t kStatusBoundsCheck = 4;  // a debug build (A2AV_CHECKS) found an index out of range
constexpr int32_t kStatusArrivalTimeout = 8;  // a source's rows did not arrive within the wait limit

// Debug builds (-DA2AV_CHECKS) check segment indices and row coordinates on
// the device before they are used: a failed check sets kStatusBoundsCheck
// in the status word and the access is skipped (nothing traps).  Other
// builds compile the checks away.
#ifdef A2AV_CHECKS
__device__ __forceinline__ bool in_bounds(bool ok, int32_t *status) {
    if (!ok) atomicOr(status, kStatusBoundsCheck);
    return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, int32_t *) { return true; }
#endif

struct SegmentTable {
    int32_t src[kMaxSegments];      // rank-major index -> first ataOut row
    int32_t dst[kMaxSegments + 1];  // expert-major index -> first permuteOut row; dst[E] = A
    int32_t tmp[kMaxSegments];      // counts in expert-major order
};

// Exclusive prefix sum of n <= 256 values in place, by one warp; returns the
// total.  Lane l owns entries [8l, 8l + 8).
__device__ __forceinline__ int64_t warp_exclusive_scan_256(int32_t *a, int n, int lane) {
    int32_t v[8];
    int64_t local = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        int i = lane * 8 + k;
        v[k] = i < n ? a[i] : 0;
        local += v[k];
    }
    int64_t inc = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int64_t t = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += t;
    }
    int64_t run = inc - local;
    int64_t total = __shfl_sync(0xffffffffu, inc, 31);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        int i = lane * 8 + k;
        if (i < n) a[i] = static_cast<int32_t>(run);
        run += v[k];
    }
    __syncwarp();
    return total;
}

// One full warp calls this.  Returns true when every count is >= 0 and the
// counts sum to A; the table is only meaningful then.
__device__ __forceinline__ bool build_segment_table(const int32_t *__restrict__ recvCounts, int W,
                                                    int e, int64_t A, SegmentTable &t, int lane) {
    const int E = W * e;
    bool bad = false;
    for (int i = lane; i < E; i += 32) {
        int32_t c = recvCounts[i];
        bad |= c < 0;
        t.src[i] = c;
        t.tmp[(i % e) * W + i / e] = c;  // segment (w = i / e, j = i % e) in expert-major slot
    }
    __syncwarp();
    bad = __any_sync(0xffffffffu, bad);
    int64_t total_r = warp_exclusive_scan_256(t.src, E, lane);
    for (int i = lane; i < E; i += 32) t.dst[i] = t.tmp[i];
    __syncwarp();
    int64_t total_e = warp_exclusive_scan_256(t.dst, E, lane);
    if (lane == 0) t.dst[E] = static_cast<int32_t>(total_e);
    __syncwarp();
    return !bad && total_r == A && total_e == A;
}

// Expert-major segment holding permuteOut row d (0 <= d < A): the last
// segment starting at or before d (empty segments share their start with the
// next one, so the search skips them).
__device__ __forceinline__ int segment_of(const SegmentTable &t, int W, int e, int32_t d) {
    int lo = 0, hi = W * e;  // invariant: dst[lo] <= d < dst[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (t.dst[mid] <= d) lo = mid;
        else hi = mid;
    }
    return lo;
}

// ataOut row feeding permuteOut row d, given its expert-major segment.
__device__ __forceinline__ int32_t source_row_in(const SegmentTable &t, int W, int e, int seg, int32_t d) {
    const int j = seg / W, w = seg % W;
    return t.src[w * e + j] + (d - t.dst[seg]);
}

// Rows a GEMM CTA multiplies come in 128-row halves of its tile, counted from
// the start of each expert group.  A half whose rows of its own group lie in
// one segment is a contiguous run of ataOut rows, so the GEMM reads it there
// directly; only halves that straddle a segment boundary need the
// expert-major copy.  Rows past the group's end belong to the next group and
// their products are discarded, so they do not count.  (Both the permute
// kernel and the GEMM call this, so they agree on which halves are copied.)
constexpr int kHalfRows = 128;

__device__ __forceinline__ bool half_in_one_segment(const SegmentTable &t, int W, int e, int32_t first,
                                                    int32_t group_end) {
    const int32_t last = min(first + kHalfRows, group_end) - 1;
    return segment_of(t, W, e, first) == segment_of(t, W, e, last);
}

// The 128-row halves of the GEMM's routed tiles that do not lie in one
// segment, which the GEMM reads from the staging copy: [first row, end row),
// end the smaller of first + 128 and the group's end, in ascending order.
// Such a half holds a segment boundary strictly inside it, and a boundary
// lies in one half only, so there are fewer than W * e <= kMaxSegments.
constexpr int kMaxStagedHalves = kMaxSegments;

struct StagedHalves {
    int32_t n;  // halves listed, or -1 when there are more than kMaxStagedHalves
    int32_t half0[kMaxExperts + 1];  // first half of each expert group; half0[e] = all halves
    int32_t warp_count[32];
    int2 span[kMaxStagedHalves];
};

// Built by the whole block (blockDim.x a multiple of 32) after the segment
// table; every block of a grid builds the same list.
__device__ __forceinline__ void list_staged_halves(const SegmentTable &t, int W, int e, StagedHalves &s) {
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32, nwarps = blockDim.x / 32;
    if (warp == 0) {
        int nh = 0;
        if (lane < e) nh = (t.dst[(lane + 1) * W] - t.dst[lane * W] + kHalfRows - 1) / kHalfRows;
        int inc = nh;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        if (lane < e) s.half0[lane] = inc - nh;
        const int all = __shfl_sync(0xffffffffu, inc, 31);
        if (lane == 0) s.half0[e] = all;
    }
    __syncthreads();
    const int total = s.half0[e];
    int base = 0;
    for (int h0 = 0; h0 < total; h0 += blockDim.x) {
        const int h = h0 + tid;
        bool staged = false;
        int first = 0, end = 0;
        if (h < total) {
            int j = 0;
            while (h >= s.half0[j + 1]) ++j;  // the group holding half h
            const int g1 = t.dst[(j + 1) * W];
            first = t.dst[j * W] + (h - s.half0[j]) * kHalfRows;
            end = min(first + kHalfRows, g1);
            staged = !half_in_one_segment(t, W, e, first, g1);
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, staged);
        if (lane == 0) s.warp_count[warp] = __popc(mask);
        __syncthreads();
        int before = base, round = 0;
        for (int w = 0; w < nwarps; ++w) {
            const int c = s.warp_count[w];
            if (w < warp) before += c;
            round += c;
        }
        const int idx = before + __popc(mask & ((1u << lane) - 1u));
        if (staged && idx < kMaxStagedHalves) s.span[idx] = make_int2(first, end);
        base += round;
        __syncthreads();  // warp_count is rewritten next round
    }
    if (tid == 0) s.n = base > kMaxStagedHalves ? -1 : base;
    __syncthreads();
}

// ataOut row feeding permuteOut row d (0 <= d < A).
__device__ __forceinline__ int32_t source_row(const SegmentTable &t, int W, int e, int32_t d) {
    return source_row_in(t, W, e, segment_of(t, W, e, d), d);
}

}  // namespace a2av
